// verify_tc_fwalk.cu -- per-channel-decay tree verification for trees of up to 256
// nodes and depth 16, dv = 128: the context product on tcgen05 tensor cores, the tree
// term by fp32 walks over each node's root path.
//
// Tree closed form (Bole summary page, "Core techniques" §1), per-channel decay:
//   o_i = H0^T (e^{G_i} * q_i) + sum_{j in anc*(i)} w_ij v_j,
//   w_ij = sum_c q_ic k_jc e^{G_ic - G_jc}
// with anc*(i) the root path of node i including i and G_i the sum of g over it.  On a
// root path i = a_0, a_1 = parent(i), ..., the pair decay of a_s is the sum of g over
// a_0 .. a_{s-1}, so one walk up the path, keeping that running sum P, gives every pair
// weight w_{i a_s} = sum_c q_ic k_{a_s c} e^{P_c} and, at the root, G_i = P.
//
// Why walks.  A root path holds at most 16 nodes, so of a 256-node tree's 256 x 256
// pair weights at most 16 per row are used (about 5 in the best-first trees of a
// large draft budget).  Each weight is a 128-term fp32 sum formed on the CUDA cores and
// the tree term sum_j w_ij v_j a 16-term fp32 sum per output: no dense score tiles, no
// bf16 split of the weights, no decay factored out of a pair (so no range limit on the
// path sums), errors at fp32 rounding.  The context term H0^T (e^{G} * q) is dense (256
// x 128 x 128 per unit) and runs on the tensor cores: D[i, c] = sum_k q~[i, k] H0[k, c]
// with q~ = e^{G} * q, A = q~ (node rows, K-major) and B = the state rows (MN-major),
// both split into bf16 hi + lo parts, passes hi.hi, hi.lo and lo.hi, fp32 accumulation
// in tensor memory (two 128-row tiles of 128 columns).
//
// Rows.  Each unit's nodes are taken in depth order (row r = the r-th node by depth,
// then index).  During the channel groups two adjacent lanes own a row, each taking 8 of
// every 16-channel group: the walk up its node's path over those channels, the partial
// pair weights (16 registers, one per path slot, summed with the neighbour lane's once
// per unit) and the q~ operand.  For the outputs a thread owns the row of its
// tensor-memory lane and half of the value channels.
//
// Copies.  A group's g (fp32 rows of 64 B, 64-byte swizzled), q and k (32 B a row) and
// 16 state rows arrive by tensor copies into one of three 40 KB staging buffers; after a
// unit's groups its v arrives the same way (channels 0-63 and 64-127, 128-byte swizzled)
// in the next two buffers.  The buffers are taken in strict rotation -- a unit's groups,
// then its two v halves, then the next unit's groups -- so each copy is requested two
// uses ahead of its readers.  A group's walk needs nothing from other threads, so the
// row warps run through the groups without meeting: each warp hands its part of the
// operands to the product thread and releases the staging buffer by mbarrier arrivals,
// and the operands alternate between two buffers.  A wait tests its phase once before
// the bounded loop: the phase has usually completed, and under the walks' shared-memory
// traffic each test costs a few hundred cycles.  The rows' weights reach the output
// threads slot-major (one slot of 32 consecutive rows per load), the tree term is summed
// in packed fp32 pairs, and the outputs go out 16 channels at a time through 2 KB of
// scratch per warp, so that a warp stores whole 64-byte row pieces.  About 180 KB of
// shared memory: one CTA of 608 threads per SM.
//
// Persistent CTAs take every grid-th (request, head) unit.  Roles (608 threads):
//   warps 0-15  rows: walks and operands (per group), outputs (per unit)
//   warp 16     tree checks, root-path lists (node indices as bytes) and the depth
//               order, up to two units ahead (two copies of the tree arrays)
//   warp 17     tensor memory; one thread issues the context products
//   warp 18     copies (one thread)
// Every wait is bounded (TV_ERR_TIMEOUT); copies and products in flight are waited for
// (bounded) before tensor memory is freed.  Malformed trees zero their rows and set
// TV_ERR_TREE.
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kFacWarpsW = 16;              // warps 0-15: half a tree row per thread
constexpr int kTreeWarpW = kFacWarpsW;      // warp 16
constexpr int kMmaWarpW = kFacWarpsW + 1;   // warp 17
constexpr int kLoadWarpW = kFacWarpsW + 2;  // warp 18
constexpr int kThreadsW = (kLoadWarpW + 1) * 32;
constexpr int kFacThreads = kFacWarpsW * 32;  // 512
constexpr int kRowsW = 256;                   // nodes per tree at most
constexpr int kSlots = 16;                    // root-path length at most
constexpr int kDvW = 128;
constexpr int kGrp = 16;                      // key channels per group
constexpr int kBoxRows = 32;                  // node rows per copy box
constexpr int kTmemColsW = 256;               // D: two 128-row tiles x 128 value channels
constexpr float kLog2eW = 1.4426950408889634f;
static_assert(kFacThreads == 2 * kRowsW, "two factor threads per tree row");
static_assert(kThreadsW == 608, "roles: 16 row warps, tree, product and copy warps");

// staging: three buffers taken in rotation; a group's copies, or half of v
constexpr int kStages = 3;
constexpr uint32_t kStageBytes = 40960;
constexpr uint32_t kSg = 0;        // g: 256 rows x 64 B (16 fp32), chunk x of row j at x ^ ((j / 2) % 4)
constexpr uint32_t kSq = 16384;    // q: 256 rows x 32 B
constexpr uint32_t kSk = 24576;    // k: 256 rows x 32 B
constexpr uint32_t kSh = 32768;    // the group's 16 state rows, 16 x 512 B
// (v: 256 rows x 128 B of 64 channels, chunk x of row j at x ^ (j % 8))
// operand buffers (two, alternating by group): the context product's operands; after a
// unit's products both hold the rows' weights (16 slots x 256 rows, fp32, slot-major) and
// the output scratch
constexpr uint32_t kPqh = 0;       // q~ hi: two 128-row tiles (K-major, no swizzle)
constexpr uint32_t kPql = 8192;    // q~ lo
constexpr uint32_t kPhh = 16384;   // state hi: two 64-channel slabs of 16 rows, MN-major
constexpr uint32_t kPhl = 20480;   // state lo
constexpr uint32_t kPBuf = 24576;  // one operand buffer
constexpr uint32_t kProdBytes = 2 * kPBuf;
constexpr uint32_t kScratch = 16384;  // output scratch after the weights, 2 KB per row warp
constexpr uint32_t kQTile = 4096;  // one 128-row tile of q~ hi or lo
constexpr uint32_t kHSlab = 2048;  // one 64-channel slab of the state rows

// Barriers.  The tree arrays come in two copies (units of even and odd index), so a
// tree barrier's phase is unit / 2; a staging buffer takes every third use, so its
// barriers' phase is use / 3; an operand buffer every second group, so its barriers'
// phase is group / 2.  A row warp arrives on a buffer's barrier once per use, and can
// reach the buffer's next use only after all sixteen have arrived.
enum {
    kWTree = 0,            // [2]: tree arrays of the unit ready
    kWTfree = 2,           // [2]: tree arrays read (row threads, products, copies: 3)
    kWStage = 4,           // [3]: a staging use landed
    kWStageFree = 7,       // [3]: a staging use read (one arrival per row warp)
    kWProd = 10,           // [2]: a group's operands written (one arrival per row warp)
    kWProdDone = 12,       // [2]: a group's products done
    kWNumBars = 14
};

enum { kWN = 0, kWOff, kWRun, kWZero, kWTiles, kWOut, kWMeta = 8 };

// Shared-memory plan, identical on host and device.
struct WalkLayout {
    uint32_t s_off, p_off, tree_off, tree_bytes, meta_off, bar_off, misc_off, total;
    __host__ __device__ WalkLayout() {
        s_off = 0;
        p_off = s_off + kStages * kStageBytes;
        tree_off = p_off + kProdBytes;
        tree_bytes = kRowsW * 16 + kRowsW + kRowsW + kRowsW * 2;  // paths, order, depths, parents
        meta_off = tree_off + 2 * tree_bytes;
        bar_off = align_up(meta_off + 2 * kWMeta * 4, 16);
        misc_off = bar_off + kWNumBars * 8;
        total = misc_off + 16 + 2 * 32 * 4 + 1024;  // tmem address, flags, depth counts; alignment
    }
};

struct WalkParams {
    VerifyArgs a;
    int expire_first_wait;  // test hook: each row warp's first wait for a copy gives up at once
};

__device__ __forceinline__ float ex2w(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float2 bf16pair(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// node index in path slot s (0 = the node itself) of a packed 16-byte path list
__device__ __forceinline__ int path_node(const uint4 &p, int s) {
    const uint32_t w = s < 4 ? p.x : s < 8 ? p.y : s < 12 ? p.z : p.w;
    return static_cast<int>((w >> (8 * (s & 3))) & 0xFFu);
}

// byte offset of 16-byte chunk x of a 64-byte row j: chunks permuted by row pair (the
// tensor copy's 64-byte swizzle), so eight rows j of distinct j % 8 fall on distinct banks
__device__ __forceinline__ uint32_t row64(int j, int x) {
    return static_cast<uint32_t>(j * 64 + ((x ^ ((j >> 1) & 3)) << 4));
}

__global__ void __launch_bounds__(kThreadsW, 1)
    verify_tc_fwalk_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_g, const WalkParams P) {
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int dk = a.dk, H = a.H, ng = dk / kGrp;
    const int units = a.B * H, G = gridDim.x;
    const int nu = (units - (int)blockIdx.x + G - 1) / G;  // units of this CTA
    auto unit_of = [&](int it) { return (int)blockIdx.x + it * G; };
    const WalkLayout L;
    uint8_t *sS = smem + L.s_off;
    uint8_t *sP = smem + L.p_off;
    auto tree_base = [&](int it) { return smem + L.tree_off + (it & 1) * L.tree_bytes; };
    auto sPath = [&](int it) { return reinterpret_cast<uint4 *>(tree_base(it)); };
    auto sOrder = [&](int it) { return tree_base(it) + kRowsW * 16; };
    auto sDep = [&](int it) { return tree_base(it) + kRowsW * 17; };
    auto sPar = [&](int it) { return reinterpret_cast<int16_t *>(tree_base(it) + kRowsW * 18); };
    auto meta = [&](int it) { return reinterpret_cast<int *>(smem + L.meta_off) + (it & 1) * kWMeta; };
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sLate = reinterpret_cast<int *>(smem + L.misc_off + 4);
    int *sCnt = reinterpret_cast<int *>(smem + L.misc_off + 16);  // per depth: count, start
    const uint32_t bar0 = ptx::smem_addr(smem + L.bar_off);
    auto bar = [&](int idx) { return bar0 + 8u * idx; };
    auto b_prod = [&](int grp) { return bar(kWProd + (grp & 1)); };
    auto b_pdone = [&](int grp) { return bar(kWProdDone + (grp & 1)); };
    auto gph = [](int grp) { return static_cast<uint32_t>((grp >> 1) & 1); };  // operand phase
    auto b_tree = [&](int it) { return bar(kWTree + (it & 1)); };
    auto b_tfree = [&](int it) { return bar(kWTfree + (it & 1)); };
    auto b_stage = [&](int use) { return bar(kWStage + use % kStages); };
    auto b_sfree = [&](int use) { return bar(kWStageFree + use % kStages); };
    auto ph = [](int it) { return static_cast<uint32_t>((it >> 1) & 1); };
    auto uph = [](int use) { return static_cast<uint32_t>((use / kStages) & 1); };
    auto stage = [&](int use) { return sS + (use % kStages) * kStageBytes; };
    const uint32_t pA = ptx::smem_addr(sP);
    auto late_now = [&]() { return *reinterpret_cast<volatile int *>(sLate) != 0; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_g);
        for (int p = 0; p < 2; ++p) {
            ptx::mbar_init(bar(kWTree + p), 1);
            ptx::mbar_init(bar(kWTfree + p), 3);
        }
        for (int b = 0; b < kStages; ++b) {
            ptx::mbar_init(bar(kWStage + b), 1);
            ptx::mbar_init(bar(kWStageFree + b), kFacWarpsW);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(kWProd + b), kFacWarpsW);
            ptx::mbar_init(bar(kWProdDone + b), 1);
        }
        ptx::fence_mbar_init();
        *sLate = 0;
    }
    if (warp == kMmaWarpW) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), kTmemColsW);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tD = *sTmem;  // lane = row of a 128-row tile, column = tile * 128 + channel

    ptx::grid_dependency_wait();  // inputs may be written by the previous kernel
    if (tid == 0) ptx::grid_launch_dependents();

    if (warp == kTreeWarpW) {
        // ================= trees: checks, root-path lists, depth order
        for (int it = 0; it < nu; ++it) {
            bool ok = true;
            if (it >= 2 && lane == 0)
                ok = !late_now() && ptx::mbar_wait(b_tfree(it - 2), ph(it - 2), kWaitLimit);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) atomicOr(sLate, 32);
                break;
            }
            const int u = unit_of(it), b = u / H, h = u % H;
            int off = 0, n = 0;
            const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
            if (!range_ok) n = 0;
            uint4 *path_s = sPath(it);
            uint8_t *ord_s = sOrder(it), *dep_s = sDep(it);
            int16_t *par_s = sPar(it);
            int *mt = meta(it);
            bool bad = false;
            int pr[8], dp[8];
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int i = lane + 32 * s;
                pr[s] = -1;
                dp[s] = 0;
                if (i < n) {
                    pr[s] = a.parent[off + i];
                    dp[s] = a.depth[off + i];
                    const bool bi = pr[s] < -1 || pr[s] >= i || dp[s] < 1 || dp[s] > a.max_depth;
                    bad = bad || bi;
                    if (bi) pr[s] = -1;  // keeps the lookups below inside the tree
                    par_s[i] = static_cast<int16_t>(pr[s]);
                    dep_s[i] = static_cast<uint8_t>(bi ? 0 : dp[s]);
                }
            }
            __syncwarp();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int i = lane + 32 * s;
                if (i < n) {
                    const int want = pr[s] < 0 ? 1 : dep_s[pr[s]] + 1;
                    bad = bad || dp[s] != want;
                }
            }
            const bool tree_bad = __any_sync(0xffffffffu, bad);
            const bool run = n > 0 && !tree_bad;
            if (run) {
                // root-path lists: the node, its parent, ... up to its root (depth entries)
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {
                    const int i = lane + 32 * s;
                    if (i < n) {
                        uint32_t w4[4] = {0u, 0u, 0u, 0u};
                        int j = i;
#pragma unroll
                        for (int sl = 0; sl < kSlots; ++sl) {
                            if (j >= 0) {
                                w4[sl >> 2] |= static_cast<uint32_t>(j) << (8 * (sl & 3));
                                j = par_s[j];
                            }
                        }
                        path_s[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
                // depth order: rank within a depth by node index, then per-depth starts
                if (lane <= kSlots) sCnt[lane] = 0;
                __syncwarp();
                int rk[8];
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const int i = lane + 32 * s;
                    const int d = i < n ? dp[s] : 0;
                    const uint32_t m = __match_any_sync(0xffffffffu, d);
                    const int base = d > 0 ? sCnt[d] : 0;
                    rk[s] = base + __popc(m & ((1u << lane) - 1u));
                    __syncwarp();
                    if (d > 0 && lane == __ffs(m) - 1) sCnt[d] = base + __popc(m);
                    __syncwarp();
                }
                const int cnt = (lane >= 1 && lane <= kSlots) ? sCnt[lane] : 0;
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                __syncwarp();
                if (lane <= kSlots) sCnt[32 + lane] = incl - cnt;
                __syncwarp();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const int i = lane + 32 * s;
                    if (i < n) ord_s[sCnt[32 + dp[s]] + rk[s]] = static_cast<uint8_t>(i);
                }
            }
            if (lane == 0) {
                if (!range_ok && h == 0) report(a.status, TV_ERR_TREE);
                if (n > 0 && tree_bad && h == 0) report(a.status, TV_ERR_TREE);
                mt[kWN] = n;
                mt[kWOff] = off;
                mt[kWRun] = run ? 1 : 0;
                mt[kWZero] = (n > 0 && tree_bad) ? 1 : 0;
                mt[kWTiles] = (n + 127) / 128;
                mt[kWOut] = 0;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_tree(it));
        }
    } else if (warp == kLoadWarpW) {
        if (lane == 0) {
            // ================= copies (one thread): staging uses in rotation -- a unit's
            // groups, then its two v halves; each use waits for the use three before it
            int U = 0;  // staging uses issued
            bool ok = true;
            auto wait_ok = [&](uint32_t b, uint32_t parity) {
                if (late_now()) return false;
                if (!ptx::mbar_wait(b, parity, kWaitLimit)) atomicOr(sLate, 64);
                return !late_now();
            };
            auto take = [&]() {  // the buffer of use U is free
                return U < kStages || wait_ok(b_sfree(U - kStages), uph(U - kStages));
            };
            for (int it = 0; it < nu && ok; ++it) {
                if (!wait_ok(b_tree(it), ph(it))) break;
                const int *mt = meta(it);
                const int n = mt[kWN], off = mt[kWOff], run = mt[kWRun];
                ptx::mbar_arrive(b_tfree(it));
                if (!run) continue;
                const int u = unit_of(it), h = u % H;
                const int rows = (n + kBoxRows - 1) / kBoxRows * kBoxRows;
                for (int g = 0; g < ng + 2 && ok; ++g, ++U) {
                    if (!take()) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ptx::smem_addr(stage(U));
                    if (g < ng) {
                        ptx::mbar_arrive_expect_tx(b_stage(U), rows * (64 + 32 + 32) + kGrp * kDvW * 4);
                        for (int r = 0; r < rows; r += kBoxRows) {
                            ptx::tma_load_3d(dst + kSg + r * 64, &tm_g, g * kGrp, h, off + r, b_stage(U));
                            ptx::tma_load_3d(dst + kSq + r * 32, &tm_q, g * kGrp, h, off + r, b_stage(U));
                            ptx::tma_load_3d(dst + kSk + r * 32, &tm_k, g * kGrp, h, off + r, b_stage(U));
                        }
                        ptx::bulk_g2s(dst + kSh, a.H0 + ((size_t)u * dk + g * kGrp) * kDvW,
                                      kGrp * kDvW * 4, b_stage(U));
                    } else {  // v channels 0-63, then 64-127
                        ptx::mbar_arrive_expect_tx(b_stage(U), rows * 128);
                        for (int r = 0; r < rows; r += kBoxRows)
                            ptx::tma_load_3d(dst + r * 128, &tm_v, (g - ng) * 64, h, off + r, b_stage(U));
                    }
                }
            }
            // every copy requested lands before the CTA's memory can go away (a buffer's
            // uses are issued one at a time, so only the last of each can be pending)
            bool drained = true;
            for (int k = 1; k <= kStages && k <= U; ++k)
                drained = ptx::mbar_wait(b_stage(U - k), uph(U - k), kWaitLimit) && drained;
            if (!drained) atomicOr(sLate, 128);
        }
    } else if (warp == kMmaWarpW) {
        if (lane == 0) {
            // ================= context products (one thread)
            int pu = 0;
            auto wait_ok = [&](uint32_t b, uint32_t parity) {
                if (late_now()) return false;
                if (!ptx::mbar_wait(b, parity, kWaitLimit)) atomicOr(sLate, 16);
                return !late_now();
            };
            constexpr uint32_t idesc = ptx::idesc_bf16_f32_bmn(128, 128);
            bool ok = true;
            for (int it = 0; it < nu && ok; ++it) {
                if (!wait_ok(b_tree(it), ph(it))) break;
                const int *mt = meta(it);
                const int run = mt[kWRun], tiles = mt[kWTiles];
                ptx::mbar_arrive(b_tfree(it));
                if (!run) continue;
                for (int g = 0; g < ng; ++g) {
                    if (!wait_ok(b_prod(pu), gph(pu))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t pb = pA + (pu & 1) * kPBuf;
                    const uint64_t bh = ptx::desc_mnmajor_sw128(pb + kPhh, kHSlab, 1024);
                    const uint64_t bl = ptx::desc_mnmajor_sw128(pb + kPhl, kHSlab, 1024);
                    for (int t = 0; t < tiles; ++t) {
                        const uint32_t d = tD + t * 128;
                        const uint64_t ah = ptx::desc_kmajor_noswizzle(pb + kPqh + t * kQTile, 128, 256);
                        const uint64_t al = ptx::desc_kmajor_noswizzle(pb + kPql + t * kQTile, 128, 256);
                        ptx::mma_bf16(d, ah, bh, idesc, g > 0 ? 1u : 0u);
                        ptx::mma_bf16(d, ah, bl, idesc, 1u);
                        ptx::mma_bf16(d, al, bh, idesc, 1u);
                    }
                    ptx::mma_commit(b_pdone(pu));
                    ++pu;
                }
            }
            // the products complete before tensor memory is freed (commits complete in order)
            if (pu > 0 && !ptx::mbar_wait(b_pdone(pu - 1), gph(pu - 1), kWaitLimit)) atomicOr(sLate, 128);
        }
    } else {
        // ================= rows (warps 0-15).  Groups: row r = ft / 2, half hf = ft % 2 of
        // every 16-channel group (8 channels: 16-byte chunks 2 hf, 2 hf + 1 of a 64-byte g
        // row, bytes 16 hf .. of a 32-byte q or k row).  Outputs: row re = (warp % 8) * 32 +
        // lane, its tensor-memory lane, and value channels 64 he .., he = warp / 8.
        const int ft = tid;
        const int hf = ft & 1, r = ft >> 1;
        const int he = warp >> 3, re = (warp & 7) * 32 + lane;
        const int qd = warp & 3, tile = (warp >> 2) & 1;  // tensor-memory lane quadrant, D tile
        int pu = 0, U = 0;  // groups handed to the product thread, staging uses read
        bool first = true;
        // the whole role: thread 0 waits (for b, then b2, where given), the barrier hands
        // the verdict, and-ed with every thread's `mine`, to all 512 threads at once
        auto sync_wait = [&](uint32_t b, uint32_t parity, bool mine, uint32_t b2 = 0u,
                             uint32_t parity2 = 0u) {
            bool ok = mine;
            if (ft == 0) {
                ok = ok && !late_now() && (b == 0u || ptx::mbar_wait(b, parity, kWaitLimit));
                if (ok && b2 != 0u) ok = ptx::mbar_wait(b2, parity2, kWaitLimit);
                if (!ok) atomicOr(sLate, 4);
            }
            return named_barrier_and(1, kFacThreads, ok);
        };
        // one warp: lane 0 waits for b (then b2, where given), the warp learns the
        // verdict.  The phases are usually complete already: one test each first.
        auto warp_wait = [&](uint32_t b, uint32_t parity, uint32_t b2, uint32_t parity2, bool expire) {
            bool ok = true;
            if (lane == 0) {
                ok = !expire && (ptx::mbar_test_wait(b, parity) ||
                                 (!late_now() && ptx::mbar_wait(b, parity, kWaitLimit)));
                if (ok && b2 != 0u)
                    ok = ptx::mbar_test_wait(b2, parity2) ||
                         (!late_now() && ptx::mbar_wait(b2, parity2, kWaitLimit));
                if (!ok) atomicOr(sLate, 8);
            }
            return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        };
        for (int it = 0; it < nu; ++it) {
            if (!sync_wait(b_tree(it), ph(it), true)) break;
            int *mt = meta(it);
            const int n = mt[kWN], off = mt[kWOff], run = mt[kWRun];
            const int u = unit_of(it), h = u % H;
            if (!run) {
                if (mt[kWZero] && r < n) {
                    float4 *o = reinterpret_cast<float4 *>(a.out + ((size_t)(off + r) * H + h) * kDvW + 64 * hf);
#pragma unroll 4
                    for (int x = 0; x < 16; ++x) o[x] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                named_barrier(1, kFacThreads);
                if (ft == 0) ptx::mbar_arrive(b_tfree(it));
                continue;
            }
            const bool active = r < n;
            const int i = active ? sOrder(it)[r] : 0;
            const int d = active ? sDep(it)[i] : 0;
            const uint4 path = active ? sPath(it)[i] : make_uint4(0u, 0u, 0u, 0u);
            const int dmax = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(d));
            float w[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s) w[s] = 0.f;
            bool ok = true;  // the same in every lane of the warp
            for (int g = 0; g < ng; ++g, ++U, ++pu) {
                // the group's copies have landed, and the operand buffer's previous products
                // (group pu - 2) are done
                if (ok)
                    ok = warp_wait(b_stage(U), uph(U), pu >= 2 ? b_pdone(pu - 2) : 0u, gph(pu - 2),
                                   first && P.expire_first_wait);
                first = false;
                if (!ok) continue;
                const uint8_t *sb = stage(U);
                uint8_t *pb = sP + (pu & 1) * kPBuf;
                float qt[8];
                if (active) {
                    // the walk up the root path: at slot s the running sum P of g over the
                    // slots below it is the pair decay of the slot's node, in base 2
                    const uint4 qh = *reinterpret_cast<const uint4 *>(sb + kSq + i * 32 + 16 * hf);
                    const uint32_t qw[4] = {qh.x, qh.y, qh.z, qh.w};
                    float qv[8], P2[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        qv[2 * e] = bf16lo(qw[e]);
                        qv[2 * e + 1] = bf16hi(qw[e]);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) P2[e] = 0.f;
#pragma unroll
                    for (int s = 0; s < kSlots; ++s) {
                        if (s >= dmax) break;
                        if (s < d) {
                            const int j = path_node(path, s);
                            const uint32_t o = row64(j, 2 * hf);
                            const float4 g0 = *reinterpret_cast<const float4 *>(sb + kSg + o);
                            const float4 g1 = *reinterpret_cast<const float4 *>(sb + kSg + (o ^ 16u));
                            const uint4 kr = *reinterpret_cast<const uint4 *>(sb + kSk + j * 32 + 16 * hf);
                            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
                            const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                            float acc = 0.f;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                acc = fmaf(qv[2 * e] * bf16lo(kw[e]), ex2w(P2[2 * e]), acc);
                                acc = fmaf(qv[2 * e + 1] * bf16hi(kw[e]), ex2w(P2[2 * e + 1]), acc);
                            }
                            w[s] += acc;
#pragma unroll
                            for (int e = 0; e < 8; ++e) P2[e] = fmaf(gv[e], kLog2eW, P2[e]);
                        }
                    }
                    // at the root P = G_i: the context product's q~ = e^{G_i} q_i, hi / lo in
                    // row r of tile r / 128 (8-row x 16-byte core matrices; this half's 8
                    // channels are the K-chunk hf)
#pragma unroll
                    for (int e = 0; e < 8; ++e) qt[e] = qv[e] * ex2w(P2[e]);
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) split_pair(qt[2 * m], qt[2 * m + 1], hi[m], lo[m]);
                    const int rr = r & 127;
                    const uint32_t qo = (r >> 7) * kQTile + (rr >> 3) * 256 + (rr & 7) * 16 + 128 * hf;
                    *reinterpret_cast<uint4 *>(pb + kPqh + qo) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(pb + kPql + qo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                {
                    // the group's 16 state rows -> hi / lo, MN-major with 128-byte swizzle:
                    // row k of slab c / 64 at k * 128, 16-byte chunk (c % 64) / 8 XOR k % 8;
                    // thread ft takes 4 channels: row ft / 32, channels 4 (ft % 32) ..
                    const int kr = ft >> 5, c4 = ft & 31;
                    const float4 x0 = *reinterpret_cast<const float4 *>(sb + kSh + kr * 512 + c4 * 16);
                    uint32_t hi[2], lo[2];
                    split_pair(x0.x, x0.y, hi[0], lo[0]);
                    split_pair(x0.z, x0.w, hi[1], lo[1]);
                    const uint32_t ho = (c4 >> 4) * kHSlab + kr * 128 + ((((c4 & 15) >> 1) ^ (kr & 7)) << 4) + (c4 & 1) * 8;
                    *reinterpret_cast<uint2 *>(pb + kPhh + ho) = make_uint2(hi[0], hi[1]);
                    *reinterpret_cast<uint2 *>(pb + kPhl + ho) = make_uint2(lo[0], lo[1]);
                }
                // this warp's operands are written and its reads of the staging buffer done
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(b_prod(pu));
                    ptx::mbar_arrive(b_sfree(U));
                }
            }
            // the two halves of a row sit in adjacent lanes: full weights in both
#pragma unroll
            for (int s = 0; s < kSlots; ++s) w[s] += __shfl_xor_sync(0xffffffffu, w[s], 1);
            // every warp through its groups (a warp that gave up makes all stop here); D is
            // full once the last group's products are done, and v has landed
            const int uv = U;  // v channels 0-63: use uv, 64-127: use uv + 1
            if (!sync_wait(b_pdone(pu - 1), gph(pu - 1), ok, b_stage(uv), uph(uv))) break;
            if (!sync_wait(b_stage(uv + 1), uph(uv + 1), true)) break;
            // the rows' weights to the output threads, through the operand buffers (free
            // now): slot s of row r at sW[s * 256 + r], read by the output threads slot by slot
            float *sW = reinterpret_cast<float *>(sP);
            if (hf == 0) {
#pragma unroll
                for (int s = 0; s < kSlots; ++s) sW[s * kRowsW + r] = w[s];
            }
            named_barrier(1, kFacThreads);
            const bool eact = re < n;
            const int ie = eact ? sOrder(it)[re] : 0;
            const int de = eact ? sDep(it)[ie] : 0;
            const uint4 pathe = eact ? sPath(it)[ie] : make_uint4(0u, 0u, 0u, 0u);
            const int dmaxe = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(de));
            ptx::tc_fence_after_sync();
            // outputs: D[re, 64 he + :] + sum_s w_s v_{path s}, 16 channels at a time from
            // this half's v.  Each piece goes through the warp's scratch (row = lane, 64 B,
            // chunks permuted by row pair) and leaves as 64-byte row pieces, 8 rows per store
            // instruction.
            uint8_t *scr = sP + kScratch + warp * 2048;
            const uint8_t *vb = stage(uv + he);
#pragma unroll 1
            for (int m4 = 0; m4 < 4; ++m4) {
                const int m = 4 * he + m4;   // 16-channel piece of the row
                const int c0 = (2 * m) & 7;  // first 16-byte chunk of the piece in a v row
                uint32_t dv[16];
                ptx::tmem_ld_x16_nowait(tD + (static_cast<uint32_t>(32 * qd) << 16) + tile * 128 + 16 * m, dv);
                ptx::tmem_wait_ld();
                float2 acc[8];  // channel pairs (2e, 2e + 1) of the piece
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] = make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1]));
                if (eact) {
#pragma unroll
                    for (int s = 0; s < kSlots; ++s) {
                        if (s >= dmaxe) break;
                        if (s < de) {
                            const int j = path_node(pathe, s);
                            const float wsv = sW[s * kRowsW + re];
                            const float2 ws = make_float2(wsv, wsv);
#pragma unroll
                            for (int x = 0; x < 2; ++x) {
                                const uint4 raw = *reinterpret_cast<const uint4 *>(vb + j * 128 + (((c0 + x) ^ (j & 7)) << 4));
                                acc[4 * x] = __ffma2_rn(ws, bf16pair(raw.x), acc[4 * x]);
                                acc[4 * x + 1] = __ffma2_rn(ws, bf16pair(raw.y), acc[4 * x + 1]);
                                acc[4 * x + 2] = __ffma2_rn(ws, bf16pair(raw.z), acc[4 * x + 2]);
                                acc[4 * x + 3] = __ffma2_rn(ws, bf16pair(raw.w), acc[4 * x + 3]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    *reinterpret_cast<float4 *>(scr + row64(lane, x)) =
                        make_float4(acc[2 * x].x, acc[2 * x].y, acc[2 * x + 1].x, acc[2 * x + 1].y);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int row = 8 * k + (lane >> 2), x = lane & 3;
                    const float4 val = *reinterpret_cast<const float4 *>(scr + row64(row, x));
                    const int node = __shfl_sync(0xffffffffu, ie, row);
                    if (32 * (warp & 7) + row < n)
                        *reinterpret_cast<float4 *>(a.out + ((size_t)(off + node) * H + h) * kDvW + 16 * m + 4 * x) = val;
                }
                __syncwarp();
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {  // this warp's reads of v done
                ptx::mbar_arrive(b_sfree(uv));
                ptx::mbar_arrive(b_sfree(uv + 1));
            }
            named_barrier(1, kFacThreads);  // D, the weights, the scratch and the tree arrays read
            if (ft == 0) ptx::mbar_arrive(b_tfree(it));
            U += 2;
        }
    }

    // ================= all roles done: report, free tensor memory
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && *sLate) report(a.status, TV_ERR_TIMEOUT);
    if (warp == kMmaWarpW) ptx::tmem_dealloc(tD, kTmemColsW);
}

// node rows of `width` elements per (node, head): dims (width, H, T), boxes of
// `box_w` elements x one head x kBoxRows nodes
bool encode_node_rows(CUtensorMap *tm, const void *base, CUtensorMapDataType dt, int esize, int width,
                      int H, int T, int box_w, CUtensorMapSwizzle swz) {
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)width * esize, (cuuint64_t)width * esize * H};
    const cuuint32_t box[3] = {(cuuint32_t)box_w, 1, (cuuint32_t)kBoxRows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_fn()(tm, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool verify_tc_fwalk_supported(const VerifyArgs &a) {
    return a.decay == TV_DECAY_DIAG && a.qkv_dtype == TV_BF16 && (a.dk == 64 || a.dk == 128) &&
           a.dv == kDvW && a.max_nodes >= 1 && a.max_nodes <= kRowsW && a.max_depth >= 1 &&
           a.max_depth <= kSlots && encode_fn() != nullptr && WalkLayout().total <= kSmemLimit;
}

cudaError_t launch_verify_tc_fwalk(const VerifyArgs &a, cudaStream_t s, bool expire_first_wait) {
    if (!verify_tc_fwalk_supported(a)) return cudaErrorNotSupported;
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv_, tg;
    // q, k: 16-channel rows; g: 16 fp32 channels, 64-byte swizzle; v: 64-channel
    // 128-byte-swizzled rows
    if (!(encode_node_rows(&tq, a.q, BF, 2, a.dk, a.H, a.T, kGrp, CU_TENSOR_MAP_SWIZZLE_NONE) &&
          encode_node_rows(&tk, a.k, BF, 2, a.dk, a.H, a.T, kGrp, CU_TENSOR_MAP_SWIZZLE_NONE) &&
          encode_node_rows(&tv_, a.v, BF, 2, kDvW, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_node_rows(&tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dk, a.H, a.T, kGrp,
                           CU_TENSOR_MAP_SWIZZLE_64B)))
        return cudaErrorInvalidValue;
    WalkParams P;
    P.a = a;
    P.expire_first_wait = expire_first_wait ? 1 : 0;
    auto kern = verify_tc_fwalk_kernel;
    cudaError_t e = configure_smem_once(kern, true);
    if (e != cudaSuccess) return e;
    const size_t smem = WalkLayout().total;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = resident_ctas(kern, kThreadsW, smem, kTmemColsW, per_sm)) != cudaSuccess)
        return e;
    const long long units = (long long)a.B * a.H;
    const long long grid = std::min<long long>(units, (long long)sms * per_sm);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreadsW), smem, s, tq, tk, tv_, tg, P);
}

}  // namespace tv
