// verify_tc_stream.cu -- scalar-decay tree verification on tcgen05 tensor cores,
// persistent: every CTA streams many (request, head) units through a two-stage
// shared-memory ring.
//
// Same arithmetic, operand layouts and error behaviour as the warp-specialized
// kernel of verify_tc.cu (tree closed form, Bole summary page, "Core techniques"
// §1; only the per-token factors are read, §2):
//   o_i = e^{G_i} (H0^T q_i) + sum_d e^{G_i - G_{anc_d(i)}} (q_i . k_{anc_d(i)}) v_{anc_d(i)}.
//
// Why a second kernel: with one CTA per unit, an SM holds the next unit's bytes in
// flight only while a CTA is still waiting for its own; once a CTA's data has
// landed it spends the rest of its life on tree checks, scores, the MMA and the
// epilogue with nothing in flight.  A launch over many units (layers folded into
// the head axis) is then bound by that idle time, not by HBM.  Here the loads of
// unit i+1 are issued while unit i is being computed.
//
// Roles, 288 threads:
//   warp 8, the producer: for each unit of the CTA, once its stage is free, issues
//     H0 as 32-row bulk copies (one mbarrier each), the q/k/v rows as TMA tiles (one
//     mbarrier) and parent/depth/g as 4-byte cp.async copies whose completion
//     arrives on the stage's tree mbarrier.  Request offsets are read 32 units
//     ahead, one unit per lane, so no load waits on another inside the loop.
//   warps 0-3 (H0 group): split each H0 chunk in place into bf16 hi/lo K-major
//     operand rows, then issue D = H0^T q on tcgen05 (M = 128, N = nodes).
//   warps 4-7 (tree group): check the tree, number the (node, ancestor) pairs, walk
//     the root paths with their decays, then form the pair scores.
//   warps 0-7: epilogue from tensor memory, then release the stage.
// Units are dealt round-robin: CTA c takes c, c + grid, c + 2 grid, ...
// Every wait is bounded; a timeout reports TV_ERR_TIMEOUT and stops the CTA after
// waiting (bounded) for the copies it has in flight.
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kStages = 2;
constexpr int kConsumers = 256;             // warps 0-7
constexpr int kThreadsS = kConsumers + 32;  // + the producer warp
constexpr int kGroup = kConsumers / 2;
constexpr int kBarsPerStage = kMaxChunks + 3;  // H0 chunks, q/k/v tiles, tree, free
constexpr int kBarIn = kMaxChunks, kBarTree = kMaxChunks + 1, kBarFree = kMaxChunks + 2;

// Shared-memory plan, identical on host and device.  Per stage: the H0 chunks (split
// in place into the A operand, later the epilogue's staging buffer), the swizzled q
// tile (B operand), the k and v rows, the tree arrays and the request's offsets.
// Shared by the stages: the per-unit scratch of the tree group, barriers, flags.
struct StreamLayout {
    uint32_t a_off, b_off, k_off, v_off, par_off, dep_off, g_off, meta_off, stage_bytes;
    uint32_t w_off, anc_off, eg_off, poff_off, pnode_off, bar_off, misc_off, total;
    __host__ __device__ StreamLayout(int dk, int dv, int npad_max, int max_depth) {
        const uint32_t swz_tile = (dk / 64) * npad_max * 128;
        a_off = 0;
        b_off = align_up(a_off + dk * dv * 4, 1024);
        k_off = align_up(b_off + swz_tile, 1024);
        v_off = align_up(k_off + npad_max * dk * 2, 1024);
        par_off = align_up(v_off + npad_max * dv * 2, 16);
        dep_off = par_off + npad_max * 4;
        g_off = dep_off + npad_max * 4;
        meta_off = g_off + npad_max * 4;
        stage_bytes = align_up(meta_off + 16, 1024);
        const uint32_t base = kStages * stage_bytes;
        w_off = base;
        anc_off = align_up(w_off + npad_max * max_depth * 4, 16);
        eg_off = align_up(anc_off + npad_max * max_depth * 4, 16);
        poff_off = align_up(eg_off + npad_max * 4, 16);
        pnode_off = align_up(poff_off + (npad_max + 1) * 4, 16);
        bar_off = align_up(pnode_off + npad_max * max_depth, 16);
        misc_off = bar_off + (kStages * kBarsPerStage + 1) * 8;
        total = align_up(misc_off + 32, 16) + 1024;  // + slack for 1024-byte base alignment
    }
};

struct StreamParams {
    VerifyArgs a;
    int npad_max;
    int tmem_cols;
};

// Bounded wait that also gives up once `abort` is set by another role.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              const volatile int *abort) {
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimit) return false;
    }
    return true;
}

template <int DV>
__global__ void __launch_bounds__(kThreadsS, 2)
    verify_tc_stream_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const StreamParams P) {
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int dk = a.dk, H = a.H, md = a.max_depth;
    const StreamLayout L(dk, DV, P.npad_max, md);
    const uint32_t slab_bytes = P.npad_max * 128;
    float *sW = reinterpret_cast<float *>(smem + L.w_off);
    int *sAnc = reinterpret_cast<int *>(smem + L.anc_off);
    float *sEG = reinterpret_cast<float *>(smem + L.eg_off);
    int *sPairOff = reinterpret_cast<int *>(smem + L.poff_off);
    uint8_t *sPairNode = smem + L.pnode_off;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sFlag = reinterpret_cast<int *>(smem + L.misc_off + 4);    // tree error (per unit)
    int *sState = reinterpret_cast<int *>(smem + L.misc_off + 8);   // progress bits (per unit)
    int *sAbort = reinterpret_cast<int *>(smem + L.misc_off + 12);  // stop the CTA
    int *sDone = reinterpret_cast<int *>(smem + L.misc_off + 16);   // units fully consumed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int units = a.B * H;
    const int my_units =
        (int)blockIdx.x < units ? (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    const int nchunks = dk / kChunkRows;
    const uint32_t chunk_bytes = kChunkRows * DV * 4;
    auto bar = [&](int s, int j) { return ptx::smem_addr(&bars[s * kBarsPerStage + j]); };
    const uint32_t bar_mma = ptx::smem_addr(&bars[kStages * kBarsPerStage]);
    enum { kH0Late = 1, kQkvLateTree = 2, kMmaOut = 4, kQkvLateMma = 8 };

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        for (int s = 0; s < kStages; ++s) {
            for (int c = 0; c < kMaxChunks; ++c) ptx::mbar_init(bar(s, c), 1);
            ptx::mbar_init(bar(s, kBarIn), 1);
            ptx::mbar_init(bar(s, kBarTree), 33);  // 32 cp.async lanes + the offsets
            ptx::mbar_init(bar(s, kBarFree), 1);
        }
        ptx::mbar_init(bar_mma, 1);
        ptx::fence_mbar_init();
        *sFlag = 0;
        *sState = 0;
        *sAbort = 0;
        *sDone = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), P.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *sTmem;

    ptx::grid_dependency_wait();  // inputs may be written by the previous kernel
    ptx::grid_launch_dependents();

    int issued = 0;  // producer lane 0: units whose copies were issued
    if (warp == kConsumers / 32) {
        // ================= producer
        int offA = 0, offB = 0;  // this lane's look-ahead: offsets of unit (i & ~31) + lane
        for (int i = 0; i < my_units; ++i) {
            if ((i & 31) == 0) {
                const int j = i + lane;
                if (j < my_units) {
                    const int bj = (int)(blockIdx.x + (unsigned)j * gridDim.x) / H;
                    offA = a.node_offsets[bj];
                    offB = a.node_offsets[bj + 1];
                }
            }
            const int off = __shfl_sync(0xffffffffu, offA, i & 31);
            const int end = __shfl_sync(0xffffffffu, offB, i & 31);
            const int s = i % kStages;
            if (i >= kStages) {
                // the consumers release unit i - kStages
                bool ok = true;
                if (lane == 0) ok = wait_or_abort(bar(s, kBarFree), ((i / kStages) - 1) & 1, sAbort);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) atomicExch(sAbort, 1);
                    break;
                }
            }
            const int u = (int)(blockIdx.x + (unsigned)i * gridDim.x);
            const int h = u % H;
            const int n = end - off;
            const bool range_ok = off >= 0 && end >= off && end <= a.T && n <= a.max_nodes;
            const bool have = range_ok && n > 0;
            uint8_t *st = smem + s * L.stage_bytes;
            if (lane == 0) {
                if (have) {
                    const float *src = a.H0 + (size_t)u * dk * DV;
                    for (int c = 0; c < nchunks; ++c) {
                        ptx::mbar_arrive_expect_tx(bar(s, c), chunk_bytes);
                        ptx::bulk_g2s(ptx::smem_addr(st + L.a_off) + c * chunk_bytes,
                                      src + c * kChunkRows * DV, chunk_bytes, bar(s, c));
                    }
                    const int npad = (n + 15) & ~15;
                    const int slabs = dk / 64;
                    ptx::mbar_arrive_expect_tx(bar(s, kBarIn), 2 * npad * dk * 2 + npad * DV * 2);
                    for (int r = 0; r < npad; r += 16) {
                        for (int sl = 0; sl < slabs; ++sl)
                            ptx::tma_load_3d(ptx::smem_addr(st + L.b_off + sl * slab_bytes + r * 128),
                                             &tm_q, sl * 64, h, off + r, bar(s, kBarIn));
                        ptx::tma_load_3d(ptx::smem_addr(st + L.k_off) + r * dk * 2, &tm_k, 0, h,
                                         off + r, bar(s, kBarIn));
                        ptx::tma_load_3d(ptx::smem_addr(st + L.v_off) + r * DV * 2, &tm_v, 0, h,
                                         off + r, bar(s, kBarIn));
                    }
                } else {
                    // nothing to verify: complete the phases without copies
                    for (int c = 0; c < nchunks; ++c) ptx::mbar_arrive(bar(s, c));
                    ptx::mbar_arrive(bar(s, kBarIn));
                }
                int *meta = reinterpret_cast<int *>(st + L.meta_off);
                meta[0] = off;
                meta[1] = n;
                meta[2] = range_ok;
            }
            if (have) {
                const uint32_t par = ptx::smem_addr(st + L.par_off);
                const uint32_t dep = ptx::smem_addr(st + L.dep_off);
                const uint32_t gg = ptx::smem_addr(st + L.g_off);
                for (int t = lane; t < n; t += 32) {
                    ptx::cp_async_4(par + 4 * t, a.parent + off + t);
                    ptx::cp_async_4(dep + 4 * t, a.depth + off + t);
                    ptx::cp_async_4(gg + 4 * t, a.g + (size_t)(off + t) * H + h);
                }
            }
            ptx::cp_async_mbar_arrive_noinc(bar(s, kBarTree));
            if (lane == 0) ptx::mbar_arrive(bar(s, kBarTree));  // the offsets above
            issued = i + 1;
        }
    } else {
        // ================= consumers
        int mma_count = 0;
        for (int i = 0; i < my_units; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (i / kStages) & 1;
            const int u = (int)(blockIdx.x + (unsigned)i * gridDim.x);
            const int h = u % H;
            uint8_t *st = smem + s * L.stage_bytes;
            uint8_t *sA = st + L.a_off;
            uint8_t *sB = st + L.b_off;
            const __nv_bfloat16 *sK = reinterpret_cast<const __nv_bfloat16 *>(st + L.k_off);
            const __nv_bfloat16 *sV = reinterpret_cast<const __nv_bfloat16 *>(st + L.v_off);
            const int *sPar = reinterpret_cast<const int *>(st + L.par_off);
            const int *sDep = reinterpret_cast<const int *>(st + L.dep_off);
            const float *sG = reinterpret_cast<const float *>(st + L.g_off);
            const int *meta = reinterpret_cast<const int *>(st + L.meta_off);

            // the unit's offsets and tree arrays
            if (tid == 0 && !wait_or_abort(bar(s, kBarTree), ph, sAbort)) atomicExch(sAbort, 1);
            if (!named_barrier_and(3, kConsumers, *(volatile int *)sAbort == 0)) break;
            const int off = meta[0], n = meta[1];
            const bool range_ok = meta[2] != 0;
            const int npad = (n + 15) & ~15;
            const bool have_nodes = range_ok && n > 0;

            if (warp < 4) {
                // ================= H0 group: split chunks as they land, then the MMA
                constexpr int kPer = DV * (kChunkRows / 8) / kGroup;
#pragma unroll
                for (int c = 0; c < kMaxChunks; ++c) {
                    if (c >= nchunks) break;
                    if (tid == 0 && !ptx::mbar_wait(bar(s, c), ph, kWaitLimit))
                        atomicOr(sState, kH0Late);
                    named_barrier(1, kGroup);
                    const bool ok = (*sState & kH0Late) == 0 && have_nodes;
                    uint8_t *chunk = sA + c * chunk_bytes;
                    float hold[kPer][8];
                    if (ok) {
                        const float *f32 = reinterpret_cast<const float *>(chunk);
#pragma unroll
                        for (int t = 0; t < kPer; ++t) {
                            const int it = tid + t * kGroup;
                            const int ch = it % DV, kq = it / DV;
#pragma unroll
                            for (int e = 0; e < 8; ++e) hold[t][e] = f32[(kq * 8 + e) * DV + ch];
                        }
                    }
                    named_barrier(1, kGroup);  // read before it is rewritten in place
                    if (ok) {
#pragma unroll
                        for (int t = 0; t < kPer; ++t) {
                            const int it = tid + t * kGroup;
                            const int ch = it % DV, kq = it / DV;
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                split_pair(hold[t][2 * e], hold[t][2 * e + 1], hi[e], lo[e]);
                            const int r_lo = DV == 64 ? 64 + ch : ch;
                            uint8_t *lo_base = DV == 64 ? chunk : chunk + 8192;
                            *reinterpret_cast<uint4 *>(chunk + (ch / 8) * 512 + kq * 128 + (ch % 8) * 16) =
                                make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            *reinterpret_cast<uint4 *>(lo_base + (r_lo / 8) * 512 + kq * 128 +
                                                       (r_lo % 8) * 16) =
                                make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        }
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before_sync();
                named_barrier(1, kGroup);
                ptx::tc_fence_after_sync();
                if (tid == 0 && have_nodes && (*sState & kH0Late) == 0) {
                    if (ptx::mbar_wait(bar(s, kBarIn), ph, kWaitLimit)) {
                        const uint32_t idesc = ptx::idesc_bf16_f32(128, npad);
                        const uint32_t b0 = ptx::smem_addr(sB);
                        for (int c = 0; c < nchunks; ++c) {
                            const uint32_t a_hi = ptx::smem_addr(sA + c * chunk_bytes);
                            const int npass = DV == 64 ? 1 : 2;
                            for (int p = 0; p < npass; ++p) {
                                const uint32_t a_op = a_hi + p * 8192;
                                for (int s2 = 0; s2 < kChunkRows / 16; ++s2) {
                                    const int kk = c * (kChunkRows / 16) + s2;
                                    const uint64_t ad =
                                        ptx::desc_kmajor_noswizzle(a_op + s2 * 256, 128, 512);
                                    const uint64_t bd = ptx::desc_kmajor_sw128(
                                        b0 + (kk / 4) * slab_bytes + (kk % 4) * 32, 1024);
                                    ptx::mma_bf16(tmem, ad, bd, idesc,
                                                  (c > 0 || p > 0 || s2 > 0) ? 1u : 0u);
                                }
                            }
                        }
                        ptx::mma_commit(bar_mma);
                        atomicOr(sState, kMmaOut);
                    } else {
                        atomicOr(sState, kQkvLateMma);
                    }
                }
            } else {
                // ================= tree group: check, pairs, root paths, scores
                const int t = tid - kGroup;
                if (have_nodes)
                    for (int j = t; j < n; j += kGroup) {
                        const int p = sPar[j];
                        bool bad = p < -1 || p >= j;
                        if (!bad) {
                            const int want = p < 0 ? 1 : sDep[p] + 1;
                            bad = sDep[j] != want || sDep[j] > md;
                        }
                        if (bad) *sFlag = 1;
                    }
                named_barrier(2, kGroup);
                const bool tree_ok = have_nodes && *sFlag == 0;
                if (tree_ok && warp == 4) {
                    // (node, ancestor) pairs numbered node by node: exclusive scan of depths
                    const int per = (n + 31) / 32;
                    int local = 0;
                    for (int q = 0; q < per; ++q) {
                        const int j = lane * per + q;
                        if (j < n) local += sDep[j];
                    }
                    int incl = local;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    int run_sum = incl - local;
                    for (int q = 0; q < per; ++q) {
                        const int j = lane * per + q;
                        if (j < n) {
                            sPairOff[j] = run_sum;
                            run_sum += sDep[j];
                        }
                    }
                    if (lane == 31) sPairOff[n] = incl;
                }
                named_barrier(2, kGroup);
                if (tree_ok) {
                    // anc_d(j), e^{G_j - G_{anc_d(j)}} and e^{G_j}
                    for (int j = t; j < n; j += kGroup) {
                        float sg = 0.f;
                        int x = j, d = 0;
                        const int p0 = sPairOff[j];
                        while (x >= 0) {
                            sAnc[p0 + d] = x;
                            sW[p0 + d] = expf(sg);
                            sPairNode[p0 + d] = static_cast<uint8_t>(j);
                            sg += sG[x];
                            x = sPar[x];
                            ++d;
                        }
                        sEG[j] = expf(sg);
                    }
                }
                if (t == 0 && have_nodes && !ptx::mbar_wait(bar(s, kBarIn), ph, kWaitLimit))
                    atomicOr(sState, kQkvLateTree);
                named_barrier(2, kGroup);
                if (tree_ok && (*sState & kQkvLateTree) == 0) {
                    pair_scores(sB, sK, sPairOff, sPairNode, sAnc, sW, n, dk, slab_bytes,
                                (warp - 4) * 4 + (lane >> 3), lane);
                }
            }

            // ================= join
            ptx::tc_fence_before_sync();
            named_barrier(3, kConsumers);
            ptx::tc_fence_after_sync();
            const int stt = *sState;
            const bool tree_ok = *sFlag == 0;
            const bool mma_out = (stt & kMmaOut) != 0;
            if (tid == 0) {
                if (!range_ok && h == 0) report(a.status, TV_ERR_TREE);
                if (have_nodes && !tree_ok && h == 0) report(a.status, TV_ERR_TREE);
                if (stt & (kH0Late | kQkvLateTree | kQkvLateMma)) report(a.status, TV_ERR_TIMEOUT);
            }
            if (have_nodes && !tree_ok)
                for (int e = tid; e < n * DV; e += kConsumers)
                    a.out[((size_t)(off + e / DV) * H + h) * DV + e % DV] = 0.f;
            bool mma_ok = true;
            if (mma_out && tid == 0) mma_ok = ptx::mbar_wait(bar_mma, mma_count & 1, kWaitLimit);
            mma_ok = named_barrier_and(3, kConsumers, mma_ok);
            if (mma_out) ++mma_count;
            if (mma_out && !mma_ok && tid == 0) report(a.status, TV_ERR_TIMEOUT);
            ptx::tc_fence_after_sync();
            const bool late = (stt & (kH0Late | kQkvLateTree | kQkvLateMma)) != 0 || !mma_ok;
            const bool run = have_nodes && tree_ok && mma_out && mma_ok && !(stt & kQkvLateTree);

            // ---- epilogue, 32 node columns at a time (as in the one-unit kernel)
            float *sXc = reinterpret_cast<float *>(sA);  // A is free once the MMAs completed
            const int quad = warp & 3, half = warp >> 2;
            const uint32_t tq = tmem + (static_cast<uint32_t>(32 * quad) << 16);
            constexpr int kQuads = DV / 4;
            for (int c0 = 0; c0 < npad && run; c0 += 32) {  // uniform bounds
                const int ncol = min(32, npad - c0);
                const int row = 32 * quad + lane;
                for (int col = half * (ncol / 2); col < (half + 1) * (ncol / 2); col += 8) {
                    float vals[8];
                    ptx::tmem_ld_x8(tq + c0 + col, vals);
#pragma unroll
                    for (int e = 0; e < 8; ++e) sXc[(col + e) * 128 + row] = vals[e];
                }
                named_barrier(3, kConsumers);
                const int ntask = min(ncol, n - c0) * kQuads;
                for (int task = tid; task < ntask; task += kConsumers) {
                    const int il = task / kQuads, c = (task % kQuads) * 4;
                    const int j = c0 + il;
                    float4 o = *reinterpret_cast<const float4 *>(sXc + il * 128 + c);
                    if (DV == 64) {
                        const float4 lo = *reinterpret_cast<const float4 *>(sXc + il * 128 + 64 + c);
                        o.x += lo.x; o.y += lo.y; o.z += lo.z; o.w += lo.w;
                    }
                    const float eg = sEG[j];
                    o.x *= eg; o.y *= eg; o.z *= eg; o.w *= eg;
                    const int dj = sDep[j], p0 = sPairOff[j];
                    for (int d = 0; d < dj; ++d) {
                        const float w = sW[p0 + d];
                        const uint2 raw = *reinterpret_cast<const uint2 *>(sV + sAnc[p0 + d] * DV + c);
                        const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
                        const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
                        o.x += w * __low2float(v01); o.y += w * __high2float(v01);
                        o.z += w * __low2float(v23); o.w += w * __high2float(v23);
                    }
                    *reinterpret_cast<float4 *>(a.out + ((size_t)(off + j) * H + h) * DV + c) = o;
                }
                ptx::tc_fence_before_sync();
                named_barrier(3, kConsumers);  // staging buffer and TMEM reused next
                ptx::tc_fence_after_sync();
            }

            // ---- release the stage; a timeout stops the CTA
            if (tid == 0) {
                *sFlag = 0;
                *sState = 0;
                if (late) atomicExch(sAbort, 1);
            }
            ptx::fence_proxy_async_smem();  // generic writes to the stage before its next copies
            ptx::tc_fence_before_sync();
            const bool cont = named_barrier_and(3, kConsumers, !late);
            ptx::tc_fence_after_sync();
            if (!cont) break;
            if (tid == 0) {
                *sDone = i + 1;
                ptx::mbar_arrive(bar(s, kBarFree));
            }
        }
    }

    // ---- teardown: copies still in flight after a stop get one more bounded wait
    __syncthreads();
    if (tid == kConsumers && *sAbort) {
        for (int i = *sDone; i < issued; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (i / kStages) & 1;
            for (int c = 0; c < nchunks; ++c) ptx::mbar_wait(bar(s, c), ph, kWaitLimit);
            ptx::mbar_wait(bar(s, kBarIn), ph, kWaitLimit);
            ptx::mbar_wait(bar(s, kBarTree), ph, kWaitLimit);
        }
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// ---------------------------------------------------------------- host side

size_t stream_smem_bytes(const VerifyArgs &a) {
    const int npad_max = (a.max_nodes + 15) & ~15;
    return StreamLayout(a.dk, a.dv, npad_max, a.max_depth).total;
}

struct DeviceInfo {
    int sms = 0;
    int smem_sm = 0;
};

DeviceInfo device_info() {
    DeviceInfo d;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    return d;
}

template <int DV>
cudaError_t launch_stream(const VerifyArgs &a, cudaStream_t s) {
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv_;
    if (!(encode_rows(&tk, a.k, BF, 2, a.dk, a.H, a.T, a.dk, CU_TENSOR_MAP_SWIZZLE_NONE) &&
          encode_rows(&tv_, a.v, BF, 2, DV, a.H, a.T, DV, CU_TENSOR_MAP_SWIZZLE_NONE) &&
          encode_rows(&tq, a.q, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B)))
        return cudaErrorInvalidValue;
    StreamParams P;
    P.a = a;
    P.npad_max = (a.max_nodes + 15) & ~15;
    P.tmem_cols = tmem_columns(P.npad_max);
    const size_t smem = stream_smem_bytes(a);
    auto kern = verify_tc_stream_kernel<DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    // resident CTAs per SM from registers, shared memory (1 KB reserved per CTA),
    // warps and tensor memory
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    const DeviceInfo d = device_info();
    const int warps = kThreadsS / 32;
    const int regs_warp = ((fa.numRegs + 7) / 8) * 8 * 32;
    int per_sm = 65536 / (regs_warp * warps);
    per_sm = min(per_sm, d.smem_sm / (int)(smem + 1024));
    per_sm = min(per_sm, 64 / warps);
    per_sm = min(per_sm, 512 / P.tmem_cols);
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const long long units = (long long)a.B * a.H;
    const long long cap = (long long)d.sms * per_sm;
    const unsigned grid = (unsigned)(units < cap ? units : cap);
    return launch_pdl(kern, dim3(grid), dim3(kThreadsS), smem, s, tq, tk, tv_, P);
}

}  // namespace

bool verify_tc_stream_supported(const VerifyArgs &a) {
    return a.decay == TV_DECAY_SCALAR && a.qkv_dtype == TV_BF16 &&
           (a.dk == 64 || a.dk == 128) && (a.dv == 64 || a.dv == 128) &&
           a.max_nodes <= kMaxNodes && stream_smem_bytes(a) <= kSmemLimit &&
           encode_fn() != nullptr;
}

bool verify_tc_stream_preferred(const VerifyArgs &a) {
    // Measured on GB300 (32 Mamba-2-like layers folded, 12288 units): 178.6 us against
    // 145.9 us for the one-unit kernel, so AUTO does not pick it yet.
    constexpr bool kFaster = false;
    if (!kFaster || !verify_tc_stream_supported(a)) return false;
    const DeviceInfo d = device_info();
    if (d.sms <= 0 || d.smem_sm <= 0) return false;
    const size_t smem = stream_smem_bytes(a) + 1024;
    const long long per_sm = std::max<long long>(1, d.smem_sm / (long long)smem);
    return (long long)a.B * a.H >= 4 * per_sm * d.sms;
}

cudaError_t launch_verify_tc_stream(const VerifyArgs &a, cudaStream_t s) {
    if (!verify_tc_stream_supported(a)) return cudaErrorNotSupported;
    return a.dv == 64 ? launch_stream<64>(a, s) : launch_stream<128>(a, s);
}

}  // namespace tv
