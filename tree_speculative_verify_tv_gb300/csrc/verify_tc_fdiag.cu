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
// Shared memory.  The key channels are taken in groups of 64: per group one slot holds
// the group's 64 state rows (32 KB, four 8 KB chunks) and one holds its g, q and k
// columns (g: 64 fp32 per node, q and k: 64 bf16 per node, 128-byte swizzled), which
// are rewritten in place as the q~ / k~ hi and lo tiles.  The next group is copied in
// once the products that read the slots are done.  About 82 KB at 64 nodes, so two
// CTAs share an SM, and one CTA's products and copies overlap the other's rewrites.
//
// Roles (288 threads):
//   warps 0-3  state chunks: read, barrier, write the hi / lo blocks (per 64 value
//              channels a block of 16 key rows, MN-major, 128-byte swizzled)
//   warps 4-7  factors: path sums G of the group's channels, range check, q~ / k~ hi
//              and lo; after the last group the weight tiles (warps 4-5: one S row per
//              thread from tensor memory), the walk for out-of-range units, and the
//              v rows past the tree cleared
//   warp 8     copies, offsets, tree checks and ancestor masks (pointer doubling in
//              shared memory), tensor memory; one thread issues the products
//   warps 0-7  epilogue: one value channel per lane, half the nodes per warp
// Every wait is bounded (TV_ERR_TIMEOUT); every copy and product in flight is waited
// for (bounded) before tensor memory is freed.  Malformed trees zero their rows and set
// TV_ERR_TREE.
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kThreadsD = 288;  // nine warps: 0-3 state, 4-7 factors, 8 copies / products
static_assert(kThreadsD == 9 * 32, "the roles below take warps 0-8, the named barriers 128 threads each");
constexpr int kDvD = 128;                               // value channels
constexpr int kGrpCh = 64;                              // key channels per group
constexpr int kChunkValsD = 2048;                       // state values per chunk
constexpr uint32_t kChunkBytesD = kChunkValsD * 4;      // 8 KB
constexpr int kChunkRowsD = kChunkValsD / kDvD;         // 16 key rows
constexpr int kChunksPerGrp = kGrpCh / kChunkRowsD;     // 4
constexpr uint32_t kGrpStateBytes = kGrpCh * kDvD * 4;  // 32 KB
constexpr float kLog2eD = 1.4426950408889634f;
constexpr float kGLimit = 69.f;  // |G| bound of the scaled factors

// Shared-memory plan, identical on host and device.  The factor slot comes first: read
// as M = 128 operands, the q~ hi and lo tiles span 16 KB from their starts, inside the
// plan for every tree size.
struct DiagLayout {
    uint32_t f_off, h_off, v_off, anc_off, par_off, jmp_off, meta_off, bar_off, misc_off, total;
    __host__ __device__ explicit DiagLayout(int np) {
        f_off = 0;                                      // q | k | g (= q~lo | k~lo)
        h_off = align_up(f_off + 4 * np * 128, 1024);   // one group of state rows
        v_off = align_up(h_off + kGrpStateBytes, 1024); // v, two 64-channel blocks
        anc_off = align_up(v_off + 2 * np * 128, 16);
        par_off = anc_off + np * 8;
        jmp_off = par_off + np * 4;
        meta_off = jmp_off + np * 4;
        bar_off = align_up(meta_off + 64, 16);
        misc_off = bar_off + 24 * 8;
        total = misc_off + 16 + 1024;  // + slack for 1024-byte base alignment
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
    constexpr uint32_t kTile = NP * 128;           // one factor tile: NP rows of 128 B
    constexpr uint32_t kSboW = (NP / 8) * 128;     // weight tiles: 8-row group step
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const DiagLayout L(NP);
    const int dk = a.dk, H = a.H, ng = dk / kGrpCh;
    uint8_t *sF = smem + L.f_off;
    uint8_t *sH = smem + L.h_off;
    uint64_t *sAnc = reinterpret_cast<uint64_t *>(smem + L.anc_off);
    int *sPar = reinterpret_cast<int *>(smem + L.par_off);
    int *sJmp = reinterpret_cast<int *>(smem + L.jmp_off);
    int *meta = reinterpret_cast<int *>(smem + L.meta_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sLate = reinterpret_cast<int *>(smem + L.misc_off + 4);  // a wait gave up
    const uint32_t bar0 = ptx::smem_addr(smem + L.bar_off);
    auto b_chunk = [&](int c) { return bar0 + 8u * c; };
    auto b_conv = [&](int c) { return bar0 + 8u * (kChunksPerGrp + c); };
    const uint32_t b_fin = bar0 + 64, b_fac = bar0 + 72, b_v = bar0 + 80, b_tree = bar0 + 88,
                   b_free = bar0 + 96, b_sfull = bar0 + 104, b_wready = bar0 + 112,
                   b_dfull = bar0 + 120;
    const uint32_t fA = ptx::smem_addr(sF);
    const uint32_t hA = ptx::smem_addr(sH);
    const uint32_t vA = ptx::smem_addr(smem + L.v_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, b = unit / H, h = unit % H;

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_g);
        for (int c = 0; c < kChunksPerGrp; ++c) {
            ptx::mbar_init(b_chunk(c), 1);
            ptx::mbar_init(b_conv(c), 4);
        }
        ptx::mbar_init(b_fin, 1);
        ptx::mbar_init(b_fac, 4);
        ptx::mbar_init(b_v, 1);
        ptx::mbar_init(b_tree, 1);
        ptx::mbar_init(b_free, 1);
        ptx::mbar_init(b_sfull, 1);
        ptx::mbar_init(b_wready, 4);
        ptx::mbar_init(b_dfull, 1);
        ptx::fence_mbar_init();
        *sLate = 0;
    }
    if (warp == 8) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), P.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *sTmem;
    const uint32_t tD = tmem;       // H0^T Q~^T + V^T W^T: lane = value channel, column = node
    const uint32_t tS = tmem + NP;  // Q~ K~^T: lane = node, column = ancestor

    ptx::grid_dependency_wait();  // inputs may be written by the previous kernel

    if (warp == 8) {
        // ================= copies, tree, products
        const float *h0 = a.H0 + (size_t)unit * dk * kDvD;
        auto issue_state = [&](int kg) {  // one group's state rows (lane 0)
            for (int c = 0; c < kChunksPerGrp; ++c) {
                ptx::mbar_arrive_expect_tx(b_chunk(c), kChunkBytesD);
                ptx::bulk_g2s(hA + c * kChunkBytesD,
                              h0 + (size_t)kg * kGrpCh * kDvD + (size_t)c * kChunkValsD,
                              kChunkBytesD, b_chunk(c));
            }
        };
        if (lane == 0) issue_state(0);  // needs no offsets
        ptx::grid_launch_dependents();
        int off = 0, n = 0;
        const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
        if (!range_ok) n = 0;
        const int npad = (n + 15) & ~15;
        auto issue_factors = [&](int kg) {  // one group's q, k and g columns (lane 0)
            if (n == 0) {
                ptx::mbar_arrive(b_fin);
                return;
            }
            ptx::mbar_arrive_expect_tx(b_fin, npad * (kGrpCh * 4 + 2 * 128));
            for (int r = 0; r < npad; r += 16) {
                ptx::tma_load_3d(fA + r * 128, &tm_q, kg * kGrpCh, h, off + r, b_fin);
                ptx::tma_load_3d(fA + kTile + r * 128, &tm_k, kg * kGrpCh, h, off + r, b_fin);
                ptx::tma_load_3d(fA + 2 * kTile + r * 256, &tm_g, kg * kGrpCh, h, off + r, b_fin);
            }
        };
        if (lane == 0) {
            issue_factors(0);
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
            // ---- products (one thread)
            bool ok = run;
            int last = 0;  // the last group whose copies were issued
            const uint32_t idn = (ptx::idesc_bf16_f32(128, 16) & ~(0x3Fu << 17)) |
                                 (static_cast<uint32_t>(npad >> 3) << 17);
            const uint32_t idm = idn | (1u << 15);  // A MN-major
            const uint32_t qh = fA, kh = fA + kTile, ql = fA + 2 * kTile, kl = fA + 3 * kTile;
            // a role that gave up (its bit in sLate) released its barriers unwritten:
            // nothing more is issued then
            auto given_up = [&]() { return *reinterpret_cast<volatile int *>(sLate) != 0; };
            for (int kg = 0; kg < ng && ok; ++kg) {
                const uint32_t ph = kg & 1;
                if (!ptx::mbar_wait(b_fac, ph, kWaitLimit)) atomicOr(sLate, 16);
                if (given_up()) {
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
                // D += H0^T Q~^T, one 16-row chunk (16 key channels) at a time
                for (int c = 0; c < kChunksPerGrp; ++c) {
                    if (!ptx::mbar_wait(b_conv(c), ph, kWaitLimit)) atomicOr(sLate, 16);
                    if (given_up()) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t ca = hA + c * kChunkBytesD;
                    const uint64_t ah = ptx::desc_mnmajor_sw128(ca, 2048, 1024);
                    const uint64_t al = ptx::desc_mnmajor_sw128(ca + 4096, 2048, 1024);
                    const uint32_t o = c * 32;
                    ptx::mma_bf16(tD, ah, ptx::desc_kmajor_sw128(qh + o, 1024), idm,
                                  (kg > 0 || c > 0) ? 1u : 0u);
                    ptx::mma_bf16(tD, ah, ptx::desc_kmajor_sw128(ql + o, 1024), idm, 1u);
                    ptx::mma_bf16(tD, al, ptx::desc_kmajor_sw128(qh + o, 1024), idm, 1u);
                }
                if (!ok) break;
                if (kg + 1 < ng) {
                    // the slots are read by the products just issued; once those are done
                    // the next group is copied in
                    ptx::mma_commit(b_free);
                    if (!ptx::mbar_wait(b_free, ph, kWaitLimit)) {
                        atomicOr(sLate, 16);
                        ok = false;
                        break;
                    }
                    issue_state(kg + 1);
                    issue_factors(kg + 1);
                    last = kg + 1;
                }
            }
            ptx::mma_commit(b_sfull);  // every product issued so far, or none
            if (ok && !ptx::mbar_wait(b_wready, 0, kWaitLimit)) {
                atomicOr(sLate, 32);
                ok = false;
            }
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
            // every copy issued lands before the CTA's memory can go away
            const uint32_t pl = last & 1;
            bool drained = true;
            for (int c = 0; c < kChunksPerGrp; ++c)
                drained = ptx::mbar_wait(b_chunk(c), pl, kWaitLimit) && drained;
            drained = ptx::mbar_wait(b_fin, pl, kWaitLimit) && drained;
            drained = ptx::mbar_wait(b_v, 0, kWaitLimit) && drained;
            if (!drained) atomicOr(sLate, 128);
        }
    } else if (warp < 4) {
        // ================= state chunks -> hi / lo blocks
        // thread t: 8-value piece t % 16 of key rows t / 16 and t / 16 + 8 of a chunk
        const int pc = tid % 16, r0 = tid / 16;
        const int g = pc / 8, cg = pc % 8;
        if (tid == 0 && !ptx::mbar_wait(b_tree, 0, kWaitLimit)) atomicOr(sLate, 2);
        named_barrier(1, 128);
        bool go = !(*sLate & 2) && meta[kMRun] != 0;
        for (int kg = 0; kg < ng && go; ++kg) {
            int c = 0;
            for (; c < kChunksPerGrp; ++c) {
                if (tid == 0) {
                    // stop when another role gave up, or when this chunk does not land
                    const bool ok = *reinterpret_cast<volatile int *>(sLate) == 0 &&
                                    ((kg == 0 && c == 0 && P.expire_first_wait)
                                         ? false  // test hook: treated as expired
                                         : ptx::mbar_wait(b_chunk(c), kg & 1, kWaitLimit));
                    if (!ok) atomicOr(sLate, 2);
                }
                named_barrier(1, 128);
                if (*sLate & 2) break;  // the chunk did not land: stop converting
                uint8_t *cp = sH + c * kChunkBytesD;
                float x[2][8];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(cp + ((r0 + 8 * t) * kDvD + pc * 8) * 4);
                    const float4 v0 = src[0], v1 = src[1];
                    x[t][0] = v0.x; x[t][1] = v0.y; x[t][2] = v0.z; x[t][3] = v0.w;
                    x[t][4] = v1.x; x[t][5] = v1.y; x[t][6] = v1.z; x[t][7] = v1.w;
                }
                named_barrier(1, 128);  // the whole chunk is read before it is rewritten
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int r = r0 + 8 * t;
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        split_pair(x[t][2 * e], x[t][2 * e + 1], hi[e], lo[e]);
                    // hi blocks: [64-channel block][16 rows][128 B]; lo blocks 4 KB further
                    uint8_t *blk = cp + g * (kChunkRowsD * 128) + r * 128 + ((cg ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(blk) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(blk + 2 * kChunkRowsD * 128) =
                        make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(b_conv(c));
            }
            if (c < kChunksPerGrp) {
                // after a failed wait the group's remaining chunks are released
                // unconverted (the outputs are not written then)
                __syncwarp();
                if (lane == 0)
                    for (; c < kChunksPerGrp; ++c) ptx::mbar_arrive(b_conv(c));
                go = false;
            }
        }
    } else if (warp < 8) {
        // ================= factors, weights (warps 4-7)
        const int t = tid - 128;
        if (t == 0 && !ptx::mbar_wait(b_tree, 0, kWaitLimit)) atomicOr(sLate, 4);
        named_barrier(2, 128);
        bool go = !(*sLate & 4) && meta[kMRun] != 0;
        const int n = meta[kMN], off = meta[kMOff];
        constexpr int kPieces = NP * 8 / 128;  // (node, 8-channel piece) items per thread
        bool wide = false;                     // a path sum outside the factor range
        for (int kg = 0; kg < ng && go; ++kg) {
            if (t == 0 && !(*reinterpret_cast<volatile int *>(sLate) == 0 &&
                            ptx::mbar_wait(b_fin, kg & 1, kWaitLimit)))
                atomicOr(sLate, 4);  // another role gave up, or the columns did not land
            named_barrier(2, 128);
            if (*sLate & 4) {
                if (lane == 0) ptx::mbar_arrive(b_fac);  // release the product thread
                go = false;
                break;
            }
            // path sums of g over the group's channels: ancestors in index order, which
            // is depth order on a root path
            const float *gs = reinterpret_cast<const float *>(sF + 2 * kTile);
            float G[kPieces][8];
#pragma unroll
            for (int u = 0; u < kPieces; ++u) {
                const int e = t + 128 * u, i = e >> 3, p = e & 7;
#pragma unroll
                for (int c = 0; c < 8; ++c) G[u][c] = 0.f;
                if (i < n) {
                    uint64_t m = sAnc[i];
                    while (m) {
                        const int j = __ffsll(static_cast<long long>(m)) - 1;
                        m &= m - 1;
                        const float4 *row = reinterpret_cast<const float4 *>(gs + j * kGrpCh + p * 8);
                        const float4 g0 = row[0], g1 = row[1];
                        G[u][0] += g0.x; G[u][1] += g0.y; G[u][2] += g0.z; G[u][3] += g0.w;
                        G[u][4] += g1.x; G[u][5] += g1.y; G[u][6] += g1.z; G[u][7] += g1.w;
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c) wide = wide || !(fabsf(G[u][c]) <= kGLimit);
                }
            }
            named_barrier(2, 128);  // every path sum is read before the g rows are rewritten
#pragma unroll
            for (int u = 0; u < kPieces; ++u) {
                const int e = t + 128 * u, i = e >> 3, p = e & 7;
                const uint32_t sw = static_cast<uint32_t>(i * 128 + ((p ^ (i & 7)) << 4));
                uint32_t qhi[4] = {0u, 0u, 0u, 0u}, qlo[4] = {0u, 0u, 0u, 0u};
                uint32_t khi[4] = {0u, 0u, 0u, 0u}, klo[4] = {0u, 0u, 0u, 0u};
                if (i < n) {
                    float qv[8], kv[8];
                    bf16x8(*reinterpret_cast<const uint4 *>(sF + sw), qv);
                    bf16x8(*reinterpret_cast<const uint4 *>(sF + kTile + sw), kv);
#pragma unroll
                    for (int c = 0; c < 8; c += 2) {
                        const float e0 = ex2f(G[u][c] * kLog2eD), e1 = ex2f(G[u][c + 1] * kLog2eD);
                        const float r0 = ex2f(-G[u][c] * kLog2eD), r1 = ex2f(-G[u][c + 1] * kLog2eD);
                        split_pair(qv[c] * e0, qv[c + 1] * e1, qhi[c / 2], qlo[c / 2]);
                        split_pair(kv[c] * r0, kv[c + 1] * r1, khi[c / 2], klo[c / 2]);
                    }
                }
                *reinterpret_cast<uint4 *>(sF + sw) = make_uint4(qhi[0], qhi[1], qhi[2], qhi[3]);
                *reinterpret_cast<uint4 *>(sF + kTile + sw) =
                    make_uint4(khi[0], khi[1], khi[2], khi[3]);
                *reinterpret_cast<uint4 *>(sF + 2 * kTile + sw) =
                    make_uint4(qlo[0], qlo[1], qlo[2], qlo[3]);
                *reinterpret_cast<uint4 *>(sF + 3 * kTile + sw) =
                    make_uint4(klo[0], klo[1], klo[2], klo[3]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_fac);
        }
        if (wide) atomicOr(&meta[kMWalk], 1);

        // ---- weights, once every product of the groups is done
        if (t == 0 && !(*reinterpret_cast<volatile int *>(sLate) == 0 &&
                        ptx::mbar_wait(b_sfull, 0, kWaitLimit)))
            atomicOr(sLate, 4);
        named_barrier(2, 128);
        go = go && !(*sLate & 4);
        const bool walk = go && meta[kMWalk] != 0;
        float *W32 = reinterpret_cast<float *>(sH);  // [NP][NP]; the state slot is free now
        if (walk) {
            // out-of-range path sums: w_ij by a walk from i to the context, the pair
            // decay e^{G_i - G_j} a running product of e^{g} (global rows, through L2)
            for (int e = t; e < NP * NP; e += 128) W32[e] = 0.f;
            named_barrier(2, 128);
            const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
            const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
            const int lch = dk / 32;
            for (int i = warp - 4; i < n; i += 4) {
                const size_t ri = ((size_t)(off + i) * H + h) * dk;
                float qv[4], f[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    qv[m] = m < lch ? __bfloat162float(q[ri + lane + 32 * m]) : 0.f;
                    f[m] = 1.f;
                }
                int j = i;  // the checked tree's parents precede their children
                while (j >= 0) {
                    const size_t rj = ((size_t)(off + j) * H + h) * dk;
                    float part = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (m < lch) part += qv[m] * __bfloat162float(k[rj + lane + 32 * m]) * f[m];
                    part = warp_sum(part);
                    if (lane == 0) W32[i * NP + j] = part;
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (m < lch) f[m] *= expf(a.g[rj + lane + 32 * m]);
                    j = sPar[j];
                }
            }
            named_barrier(2, 128);
        }
        if (go && warp >= 6) {
            // rows npad > j >= n of v (another request's, or zero past the end) meet zero
            // weights; clear them so that no non-finite value gets in
            bool vok = true;
            if (lane == 0) vok = ptx::mbar_wait(b_v, 0, kWaitLimit);
            vok = __shfl_sync(0xffffffffu, vok ? 1 : 0, 0) != 0;
            if (!vok) {
                if (lane == 0) atomicOr(sLate, 8);
            } else {
                const int npad = (n + 15) & ~15;
                for (int e = (warp - 6) * 32 + lane; e < (npad - n) * 16; e += 64) {
                    const int jr = n + e / 16, mb = (e / 8) % 2, piece = e % 8;
                    *reinterpret_cast<uint4 *>(smem + L.v_off + mb * kTile + jr * 128 + piece * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        if (go && warp < 6 && 32 * (warp - 4) < NP) {
            // weight tiles: row i = node (thread), columns = ancestors, K-major without
            // swizzle (8-row x 16-byte core matrices), hi at the slot start, lo after it
            const int i = 32 * (warp - 4) + lane;
            const uint64_t m = i < NP ? sAnc[i] : 0ull;
            constexpr int CW = NP < 32 ? NP : 32;  // columns per pass
            if (!walk) ptx::tc_fence_after_sync();
#pragma unroll
            for (int cb = 0; cb < NP; cb += CW) {
                uint32_t sr[CW];
                if (!walk) {
                    tmem_ld_n<CW>(tS + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + cb, sr);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int jj = 0; jj < CW; ++jj)
                        sr[jj] = i < NP ? __float_as_uint(W32[i * NP + cb + jj]) : 0u;
                }
                uint32_t whi[CW / 2], wlo[CW / 2];
#pragma unroll
                for (int jj = 0; jj < CW; jj += 2) {
                    const float wa = ((m >> (cb + jj)) & 1ull) ? __uint_as_float(sr[jj]) : 0.f;
                    const float wb =
                        ((m >> (cb + jj + 1)) & 1ull) ? __uint_as_float(sr[jj + 1]) : 0.f;
                    split_pair(wa, wb, whi[jj / 2], wlo[jj / 2]);
                }
                if (i < NP) {
                    uint8_t *wh = sF + (i / 8) * kSboW + (i % 8) * 16 + (cb / 8) * 128;
                    uint8_t *wl = wh + NP * NP * 2;
#pragma unroll
                    for (int cc = 0; cc < CW / 8; ++cc) {
                        *reinterpret_cast<uint4 *>(wh + cc * 128) = make_uint4(
                            whi[4 * cc], whi[4 * cc + 1], whi[4 * cc + 2], whi[4 * cc + 3]);
                        *reinterpret_cast<uint4 *>(wl + cc * 128) = make_uint4(
                            wlo[4 * cc], wlo[4 * cc + 1], wlo[4 * cc + 2], wlo[4 * cc + 3]);
                    }
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
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 8) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// ---------------------------------------------------------------- host side

int fdiag_np(const VerifyArgs &a) { return a.max_nodes <= 16 ? 16 : a.max_nodes <= 32 ? 32 : 64; }

template <int NP>
cudaError_t launch_fdiag_t(const VerifyArgs &a, bool expire, cudaStream_t s) {
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv_, tg;
    // q, k: 64-channel K-major operand boxes; v: MN-major blocks of 64 channels; g: 64
    // fp32 channels per node, dense rows
    if (!(encode_rows(&tq, a.q, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tk, a.k, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tv_, a.v, BF, 2, kDvD, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dk, a.H, a.T, 64,
                      CU_TENSOR_MAP_SWIZZLE_NONE)))
        return cudaErrorInvalidValue;
    DiagParams P;
    P.a = a;
    P.tmem_cols = tmem_columns(2 * NP);
    P.expire_first_wait = expire ? 1 : 0;
    auto kern = verify_tc_fdiag_kernel<NP>;
    cudaError_t e = configure_smem_once(kern, true);
    if (e != cudaSuccess) return e;
    const size_t smem = DiagLayout(NP).total;
    return launch_pdl(kern, dim3((unsigned)(a.B * a.H)), dim3(kThreadsD), smem, s, tq, tk, tv_, tg,
                      P);
}

}  // namespace

bool verify_tc_fdiag_supported(const VerifyArgs &a) {
    return a.decay == TV_DECAY_DIAG && a.qkv_dtype == TV_BF16 && (a.dk == 64 || a.dk == 128) &&
           a.dv == kDvD && a.max_nodes >= 1 && a.max_nodes <= 64 && encode_fn() != nullptr &&
           DiagLayout(fdiag_np(a)).total <= kSmemLimit;
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
