// verify_tc_fused.cu -- scalar-decay tree verification with all three products of a
// (request, head) unit on tcgen05 tensor cores, one unit per CTA.
//
// Tree closed form (Bole summary page, "Core techniques" §1), scalar decay:
//   o_i = e^{G_i} (H0^T q_i) + sum_{j in anc*(i)} e^{G_i - G_j} (q_i . k_j) v_j
// with anc*(i) the root path of node i including i and G_i the sum of g over it.
// Only the per-token factors are read (§2); no per-node state is formed.
//
// Products, accumulators in tensor memory:
//   context  D_C = A^T q with A = the state rows split into bf16 hi and lo parts and
//            stacked along M: D_C[c][i] = sum_r hi(H0[r][c]) q_i[r] (rows 0-63) and
//            D_C[64+c][i] = sum_r lo(H0[r][c]) q_i[r] (rows 64-127), per 64 channels
//   scores   D_S[i][j] = q_i . k_j  (A = the q tile read as M = 128 rows; rows past
//            the nodes are never read)
//   tree     D_T[c][i] = sum_j v_j[c] W[i][j] with W[i][j] = e^{G_i-G_j} D_S[i][j] on
//            root paths (j in anc*(i)), else 0, in bf16 hi + lo parts
//   o_i[c]  = e^{G_i} (D_C[c][i] + D_C[64+c][i]) + D_T[c][i]
// hi(x) keeps the upper 16 bits of x (exact); lo(x) = bf16(x - hi(x)), so
// |x - hi - lo| <= 2^-16 |x|.  q, k and v are bf16, so the products are exact and
// accumulate in fp32.
//
// The state lands as contiguous chunks of 2048 values (32 key rows at dv = 64, 16
// at dv = 128) by bulk copy; warps 0-3 rewrite each chunk in place into the tensor
// core's operand: per 64 channels a block of hi rows and a block of lo rows
// (128-byte swizzled, MN-major: a row holds one key channel's 64 values), so no
// transpose is needed.  For dv = 64 without a pending commit the parts go to tensor
// memory instead (the A operand of the context product: one thread per lane, lanes
// 0-63 the hi parts and 64-127 the lo parts of the 64 value channels, packed along the
// key rows), which saves the in-place barrier and the operand's shared-memory reads.
//
// Roles (256 threads):
//   warps 0-3  chunk copies (thread 0); per chunk (per pair of chunks with a pending
//              commit): read, apply the pending commit (tv_commit_verify: H <-
//              e^{G_L} H + sum_m a_m v_m^T), barrier, write the hi / lo blocks, hand
//              the chunks to the products, then write the updated rows back to HBM
//              (256-bit stores where the state allows)
//   warp 4     offsets, q/k/v tile copies, tree checks, path sums G (pointer
//              doubling over the warp, lane = node), ancestor masks, e^{G_i}; the
//              weights from D_S into the weight tiles (its tensor-memory quadrant
//              holds the score rows)
//   warp 5     the pending path (commit + verify): checks, suffix decays, factor rows
//   warp 7     tensor-memory owner; one thread issues the products
//   all        epilogue: warps of quadrants 2-3 pass the lo rows of D_C through
//              shared memory to those of quadrants 0-1, which form o and store it
// Every wait is bounded (TV_ERR_TIMEOUT); every copy and product in flight is
// waited for (bounded) before tensor memory is freed.  Malformed trees zero their
// rows and set TV_ERR_TREE.
#include "greedy_walk.cuh"
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kThreadsF = 256;
constexpr int kChunkVals = 2048;  // state values per copied chunk (8 KB)
constexpr uint32_t kChunkBytes = kChunkVals * 4;
constexpr int kMaxChunksF = 8;    // dk * dv <= 16384
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory plan, identical on host and device.  The q tile comes first: read
// as an M = 128 operand it spans 16 KB from each slab start, all inside the plan.
struct FusedLayout {
    uint32_t q_off, k_off, v_off, whi_off, wlo_off, eg_off, meta_off, pk16_off, pv16_off,
        pa_off, pvv_off, bar_off, misc_off, acc_off, accf_off, h_off, total;
    // pd: the pending path's depth bound (commit + verify); an: the previous tree's node
    // bound when its greedy walk runs here (accept + commit + verify), else 0
    __host__ __device__ FusedLayout(int dk, int dv, int np, int pd, int an = 0) {
        const uint32_t tile = (dk / 64) * np * 128;
        q_off = 0;
        k_off = align_up(q_off + tile, 1024);
        v_off = align_up(k_off + tile, 1024);
        whi_off = align_up(v_off + (dv / 64) * np * 128, 128);
        wlo_off = whi_off + np * np * 2;
        eg_off = align_up(wlo_off + np * np * 2, 16);
        meta_off = eg_off + np * 4;
        pk16_off = align_up(meta_off + 64, 16);
        pv16_off = pk16_off + pd * dk * 2;
        pa_off = align_up(pv16_off + pd * dv * 2, 16);
        pvv_off = pa_off + pd * dk * 4;
        bar_off = align_up(pvv_off + pd * dv * 4, 16);
        misc_off = bar_off + (kMaxChunksF * 2 + 8) * 8;
        // accept mode: the walk's parent, draft and target rows and path, then every
        // node's k and v rows (bf16), prefetched while the walk runs
        acc_off = align_up(misc_off + 16, 16);
        accf_off = acc_off + align_up((3 * an + kMaxDepth) * 4, 16);
        h_off = align_up(accf_off + an * (dk + dv) * 2, 1024);
        total = h_off + dk * dv * 4 + 1024;  // + slack for 1024-byte base alignment
    }
};

// metadata words
enum { kMetaN = 0, kMetaOff, kMetaRun, kMetaZero, kMetaPL, kMetaAlpha, kMetaPBad, kMetaHave };

struct FusedParams {
    VerifyArgs a;
    PendingArgs pend;  // commit + verify only
    float *H_w;        // state rows written back (commit + verify only)
    int wb32;          // H_w is 32-byte aligned: the write-back uses 256-bit stores
    // accept + commit + verify: the pending path is the greedy walk of the previous tree
    // (pend's tree), which the head-0 block of each request also writes out
    int acc;
    const int32_t *acc_draft, *acc_target, *acc_root;
    int32_t *acc_len, *acc_path, *acc_bonus;
    int tmem_cols;
    int wave;               // CTAs resident at once (units one wave ahead are prefetched)
    int expire_first_wait;  // test hook: the first wait for a state chunk gives up at once
};

// 8 floats to a 32-byte aligned global address in one 256-bit store
__device__ __forceinline__ void st_global_v8(float *p, const float (&x)[8]) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(x[0]),
                 "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7])
                 : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 8)
        ptx::tmem_ld_x8_nowait(taddr, r);
    else if constexpr (N == 16)
        ptx::tmem_ld_x16_nowait(taddr, r);
    else
        ptx::tmem_ld_x32_nowait(taddr, r);
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int DV, int NP, bool PEND>
__global__ void __launch_bounds__(kThreadsF, PEND ? 3 : 4)
    verify_tc_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const FusedParams P) {
    constexpr int MG = DV / 64;          // 64-channel groups
    constexpr int R = kChunkVals / DV;   // key rows per chunk: 32 or 16
    constexpr uint32_t kColT = MG * NP;  // tree columns, shared with the scores
    // dv = 64 without a pending commit: the state's hi / lo parts go to tensor memory (A
    // operand of the context product; lanes 0-63 hi, 64-127 lo of the 64 value
    // channels), R / 2 columns a chunk, so a chunk is never rewritten in place
    constexpr bool kStateTmem = DV == 64 && !PEND;
    constexpr uint32_t kColA = 2 * MG * NP;
    constexpr int cpr = DV / 8;          // 8-value pieces per state row
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int dk = a.dk, H = a.H;
    const int pd = PEND ? P.pend.max_depth : 0;
    const FusedLayout L(dk, DV, NP, pd, PEND && P.acc ? P.pend.max_nodes : 0);
    const int nch = dk / R;  // chunks
    const uint32_t tile_slab = NP * 128;
    int *meta = reinterpret_cast<int *>(smem + L.meta_off);
    float *sEG = reinterpret_cast<float *>(smem + L.eg_off);
    uint8_t *sH = smem + L.h_off;
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sLate = reinterpret_cast<int *>(smem + L.misc_off + 4);  // a wait gave up
    const uint32_t bar_base = ptx::smem_addr(smem + L.bar_off);
    auto b_chunk = [&](int c) { return bar_base + 8u * c; };
    auto b_conv = [&](int c) { return bar_base + 8u * (kMaxChunksF + c); };
    const uint32_t b_qkv = bar_base + 8u * (2 * kMaxChunksF);
    const uint32_t b_sfull = b_qkv + 8, b_wready = b_qkv + 16, b_dfull = b_qkv + 24,
                   b_pend = b_qkv + 32, b_final = b_qkv + 40, b_issue = b_qkv + 48;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, b = unit / H, h = unit % H;

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        for (int c = 0; c < nch; ++c) {
            ptx::mbar_init(b_chunk(c), 1);
            ptx::mbar_init(b_conv(c), 4);
        }
        ptx::mbar_init(b_qkv, 1);
        ptx::mbar_init(b_sfull, 1);
        ptx::mbar_init(b_wready, 1);
        ptx::mbar_init(b_dfull, 1);
        ptx::mbar_init(b_pend, 1);
        ptx::mbar_init(b_final, 1);
        ptx::mbar_init(b_issue, 1);
        ptx::fence_mbar_init();
        *sLate = 0;
    }
    if (warp == 7) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), P.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *sTmem;

    ptx::grid_dependency_wait();  // inputs may be written by the previous kernel
    const float *hsrc = (PEND ? P.H_w : a.H0) + (size_t)unit * dk * DV;
    auto copy_state = [&]() {
        for (int c = 0; c < nch; ++c) {
            ptx::mbar_arrive_expect_tx(b_chunk(c), kChunkBytes);
            ptx::bulk_g2s(ptx::smem_addr(sH) + c * kChunkBytes, hsrc + (size_t)c * kChunkVals,
                          kChunkBytes, b_chunk(c));
        }
    };
    // with a pending commit the state is copied once the pending path's loads are out
    // (below), so that they do not queue behind every block's state
    if (!PEND && tid == 0) copy_state();
    // the state of the unit that starts about one wave later goes to L2 now, so its
    // CTA finds it there (same bytes, fetched earlier)
    if (tid == 32 && P.wave > 0 && unit + P.wave < a.B * H)
        ptx::prefetch_l2((PEND ? P.H_w : a.H0) + (size_t)(unit + P.wave) * dk * DV,
                         dk * DV * 4);
    ptx::grid_launch_dependents();

    if (warp < 4) {
        // ================= state chunks: read, (pending commit), rewrite as hi / lo blocks
        // thread t: 8-value piece t % cpr of rows t / cpr and t / cpr + 128 / cpr
        const int pc = tid % cpr, r0 = tid / cpr;
        constexpr int rstep = 128 / cpr;  // 16 (dv = 64) or 8 (dv = 128)
        constexpr int kRows = R / rstep;  // rows per thread per chunk: 2
        const int g = pc / 8, cg = pc % 8;
        int pL = 0;
        float alpha = 1.f;
        bool run_chunks = true;
        if constexpr (PEND) {
            bool ok = true;
            if (tid == 0) {
                // the state copies follow the pending path's loads (issued by warp 5)
                if (!ptx::mbar_wait(b_issue, 0, kWaitLimit)) atomicOr(sLate, 1);
                copy_state();
                ok = *reinterpret_cast<volatile int *>(sLate) == 0 &&
                     ptx::mbar_wait(b_pend, 0, kWaitLimit);
                if (!ok) atomicOr(sLate, 1);
            }
            // the verdict of thread 0, handed to the four warps by the barrier itself
            run_chunks = named_barrier_and(1, 128, ok);
            pL = meta[kMetaPL];
            alpha = __int_as_float(meta[kMetaAlpha]);
        }
        const float *pa = reinterpret_cast<const float *>(smem + L.pa_off);
        const float *pvv = reinterpret_cast<const float *>(smem + L.pvv_off);
        int c = 0;
        constexpr int CPI = (PEND && !kStateTmem) ? 2 : 1;  // chunks per step
        for (; c < nch && run_chunks; c += CPI) {
            bool ok = true;
            if (tid == 0) {
                ok = (c == 0 && P.expire_first_wait)
                         ? false  // test hook: treated as expired
                         : ptx::mbar_wait(b_chunk(c), 0, kWaitLimit);
                if (CPI == 2 && ok) ok = ptx::mbar_wait(b_chunk(c + 1), 0, kWaitLimit);
                if (!ok) atomicOr(sLate, 2);
            }
            if (!named_barrier_and(1, 128, ok)) break;  // the chunk did not land: stop converting
            if constexpr (kStateTmem) {
                // thread = tensor-memory lane: value channel 32 (warp & 1) + lane, the hi part
                // (warps 0-1) or the lo part (warps 2-3) of its R key rows, packed in pairs
                // along the rows (the A operand layout)
                const float *cpf = reinterpret_cast<const float *>(sH + c * kChunkBytes) +
                                   32 * (warp & 1) + lane;
                uint32_t pk[R / 2];
#pragma unroll
                for (int m = 0; m < R / 2; ++m) {
                    const float x0 = cpf[(2 * m) * DV], x1 = cpf[(2 * m + 1) * DV];
                    if (warp < 2) {
                        pk[m] = __byte_perm(__float_as_uint(x0), __float_as_uint(x1), 0x7632);
                    } else {
                        uint32_t hi;
                        split_pair(x0, x1, hi, pk[m]);
                    }
                }
                static_assert(!kStateTmem || R / 2 == 16, "dv = 64: 32 key rows a chunk");
                ptx::tmem_st_x16(tmem + kColA + c * (R / 2) + (static_cast<uint32_t>(32 * warp) << 16),
                                 reinterpret_cast<const uint32_t (&)[16]>(pk));
                ptx::tmem_wait_st();
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(b_conv(c));
                continue;
            }
            float x[CPI][kRows][8];
#pragma unroll
            for (int cc = 0; cc < CPI; ++cc)
#pragma unroll
                for (int t = 0; t < kRows; ++t) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        sH + (c + cc) * kChunkBytes + ((r0 + rstep * t) * DV + pc * 8) * 4);
                    const float4 v0 = src[0], v1 = src[1];
                    x[cc][t][0] = v0.x; x[cc][t][1] = v0.y; x[cc][t][2] = v0.z; x[cc][t][3] = v0.w;
                    x[cc][t][4] = v1.x; x[cc][t][5] = v1.y; x[cc][t][6] = v1.z; x[cc][t][7] = v1.w;
                }
            if (PEND && pL > 0) {
                // the pending rank-pL update on these rows (written back to the state
                // once the chunks are handed to the products)
#pragma unroll
                for (int cc = 0; cc < CPI; ++cc)
#pragma unroll
                    for (int t = 0; t < kRows; ++t)
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[cc][t][e] *= alpha;
                for (int m = 0; m < pL; ++m) {
                    const float4 va = *reinterpret_cast<const float4 *>(pvv + m * DV + pc * 8);
                    const float4 vb = *reinterpret_cast<const float4 *>(pvv + m * DV + pc * 8 + 4);
                    const float vm[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
                    for (int cc = 0; cc < CPI; ++cc)
#pragma unroll
                        for (int t = 0; t < kRows; ++t) {
                            const float am = pa[m * dk + (c + cc) * R + r0 + rstep * t];
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[cc][t][e] += am * vm[e];
                        }
                }
            }
            named_barrier(1, 128);  // the whole chunk is read before it is rewritten
#pragma unroll
            for (int cc = 0; cc < CPI; ++cc)
#pragma unroll
                for (int t = 0; t < kRows; ++t) {
                    const int r = r0 + rstep * t;
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        split_pair(x[cc][t][2 * e], x[cc][t][2 * e + 1], hi[e], lo[e]);
                    uint8_t *blk = sH + (c + cc) * kChunkBytes + g * (2 * R * 128) + r * 128 +
                                   ((cg ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(blk) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(blk + R * 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                for (int cc = 0; cc < CPI; ++cc) ptx::mbar_arrive(b_conv(c + cc));
            if (PEND && pL > 0) {
                // a thread's 8 values of a row fill one 32-byte sector: one 256-bit store
                // where the state is 32-byte aligned, else two 128-bit stores
#pragma unroll
                for (int cc = 0; cc < CPI; ++cc) {
                    float *Hw = P.H_w + ((size_t)unit * dk + (c + cc) * R) * DV + pc * 8;
#pragma unroll
                    for (int t = 0; t < kRows; ++t) {
                        float *dst = Hw + (r0 + rstep * t) * DV;
                        if (P.wb32) {
                            st_global_v8(dst, x[cc][t]);
                        } else {
                            reinterpret_cast<float4 *>(dst)[0] =
                                make_float4(x[cc][t][0], x[cc][t][1], x[cc][t][2], x[cc][t][3]);
                            reinterpret_cast<float4 *>(dst)[1] =
                                make_float4(x[cc][t][4], x[cc][t][5], x[cc][t][6], x[cc][t][7]);
                        }
                    }
                }
            }
        }
        // after a failed wait the remaining chunks are released unconverted, so the
        // product thread does not wait on them (the outputs are not written then)
        __syncwarp();
        if (lane == 0)
            for (; c < nch; ++c) ptx::mbar_arrive(b_conv(c));
    } else if (warp == 4) {
        // ================= offsets, tiles, tree, weights
        int off = 0, n = 0;
        const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
        if (!range_ok) n = 0;
        const int npad = (n + 15) & ~15;
        if (lane == 0) {
            if (n == 0) {
                ptx::mbar_arrive(b_qkv);  // nothing to copy
            } else {
                ptx::mbar_arrive_expect_tx(b_qkv, npad * (2 * dk * 2 + DV * 2));
                const uint32_t qa = ptx::smem_addr(smem + L.q_off);
                const uint32_t ka = ptx::smem_addr(smem + L.k_off);
                const uint32_t va = ptx::smem_addr(smem + L.v_off);
                for (int r = 0; r < npad; r += 16) {
                    for (int sb = 0; sb < dk / 64; ++sb) {
                        ptx::tma_load_3d(qa + sb * tile_slab + r * 128, &tm_q, sb * 64, h, off + r,
                                         b_qkv);
                        ptx::tma_load_3d(ka + sb * tile_slab + r * 128, &tm_k, sb * 64, h, off + r,
                                         b_qkv);
                    }
#pragma unroll
                    for (int gg = 0; gg < MG; ++gg)
                        ptx::tma_load_3d(va + gg * tile_slab + r * 128, &tm_v, gg * 64, h, off + r,
                                         b_qkv);
                }
            }
        }
        // tree rows (lane = node), checks, path sums and ancestor masks
        const bool valid = lane < n;
        int par = 0, dep = 0;
        float gv = 0.f;
        if (valid) {
            par = a.parent[off + lane];
            dep = a.depth[off + lane];
            gv = a.g[(size_t)(off + lane) * H + h];
        }
        bool bad = valid && (par < -1 || par >= lane);
        const int pdep = __shfl_sync(0xffffffffu, dep, par >= 0 && par < 32 ? par : 0);
        bad = bad || (valid && (dep != (par < 0 ? 1 : pdep + 1) || dep > a.max_depth));
        const bool tree_bad = __any_sync(0xffffffffu, bad);
        float Gs = valid ? gv : 0.f;
        uint32_t anc = valid ? (1u << lane) : 0u;
        int jmp = (valid && !tree_bad) ? par : -1;
        // pointer doubling: after round r a node covers 2^{r+1} nodes of its path
        for (int r = 0; r < 5 && __any_sync(0xffffffffu, jmp >= 0); ++r) {
            const int src = jmp >= 0 ? jmp : 0;
            const float Gj = __shfl_sync(0xffffffffu, Gs, src);
            const uint32_t aj = __shfl_sync(0xffffffffu, anc, src);
            const int jj = __shfl_sync(0xffffffffu, jmp, src);
            if (jmp >= 0) {
                Gs += Gj;
                anc |= aj;
                jmp = jj;
            }
        }
        if (lane < NP) sEG[lane] = valid ? expf(Gs) : 0.f;
        const bool run = n > 0 && !tree_bad;
        if (lane == 0) {
            if (!range_ok && h == 0) report(a.status, TV_ERR_TREE);
            if (n > 0 && tree_bad && h == 0) report(a.status, TV_ERR_TREE);
            meta[kMetaN] = n;
            meta[kMetaOff] = off;
            meta[kMetaRun] = run ? 1 : 0;
            meta[kMetaZero] = (n > 0 && tree_bad) ? 1 : 0;
        }
        bool got = true;
        if (n > 0) {
            if (lane == 0) got = ptx::mbar_wait(b_qkv, 0, kWaitLimit);
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got && lane == 0) atomicOr(sLate, 4);
        }
        if (run && got) {
            // rows npad > j >= n of v (another request's, or zero past the end) meet zero
            // weights; clear them so that no non-finite value gets in
            uint8_t *sv = smem + L.v_off;
            for (int e = lane; e < (npad - n) * 8 * MG; e += 32) {
                const int jr = n + e / (8 * MG), gg = (e / 8) % MG, piece = e % 8;
                *reinterpret_cast<uint4 *>(sv + gg * tile_slab + jr * 128 + piece * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            bool sok = true;
            if (lane == 0) sok = ptx::mbar_wait(b_sfull, 0, kWaitLimit);
            sok = __shfl_sync(0xffffffffu, sok ? 1 : 0, 0) != 0;
            if (sok) {
                ptx::tc_fence_after_sync();
                uint32_t sr[NP];
                tmem_ld_cols<NP>(tmem + kColT, sr);
                ptx::tmem_wait_ld();
                const float G2 = Gs * kLog2e;
                uint32_t whi[NP / 2], wlo[NP / 2];
#pragma unroll
                for (int jj = 0; jj < NP; jj += 2) {
                    const float G2a = __shfl_sync(0xffffffffu, G2, jj);
                    const float G2b = __shfl_sync(0xffffffffu, G2, jj + 1);
                    float wa = 0.f, wb = 0.f;
                    if ((anc >> jj) & 1u) wa = __uint_as_float(sr[jj]) * ex2_approx(G2 - G2a);
                    if ((anc >> (jj + 1)) & 1u)
                        wb = __uint_as_float(sr[jj + 1]) * ex2_approx(G2 - G2b);
                    split_pair(wa, wb, whi[jj / 2], wlo[jj / 2]);
                }
                if (lane < NP) {
                    constexpr uint32_t kSboW = (NP / 8) * 128;
                    uint8_t *wh = smem + L.whi_off + (lane / 8) * kSboW + (lane % 8) * 16;
                    uint8_t *wl = smem + L.wlo_off + (lane / 8) * kSboW + (lane % 8) * 16;
#pragma unroll
                    for (int cc = 0; cc < NP / 8; ++cc) {
                        *reinterpret_cast<uint4 *>(wh + cc * 128) = make_uint4(
                            whi[4 * cc], whi[4 * cc + 1], whi[4 * cc + 2], whi[4 * cc + 3]);
                        *reinterpret_cast<uint4 *>(wl + cc * 128) = make_uint4(
                            wlo[4 * cc], wlo[4 * cc + 1], wlo[4 * cc + 2], wlo[4 * cc + 3]);
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before_sync();
            } else if (lane == 0) {
                atomicOr(sLate, 8);
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_wready);
    } else if (warp == 5 && PEND) {
        // ================= the pending path: in range, a root path of the previous tree
        const PendingArgs &pa = P.pend;
        const int mdp = pa.max_depth;
        int poff = 0, pn = 0;
        const bool prange = request_range(pa.node_offsets, b, pa.T, pa.max_nodes, poff, pn);
        int Lq, pm;
        bool pbad;
        const int k8 = dk / 8, v8 = DV / 8;
        const __nv_bfloat16 *pk = static_cast<const __nv_bfloat16 *>(pa.k);
        const __nv_bfloat16 *pv = static_cast<const __nv_bfloat16 *>(pa.v);
        float gl = 0.f;  // accept mode: lane i holds node i's decay
        if (P.acc) {
            // every node's factor rows and decay, requested now so that they arrive with
            // the tree arrays below: the path's rows are then in shared memory once the
            // walk has found it (the previous tree has at most 32 nodes here)
            const int nacc = prange ? pn : 0;
            const uint32_t fk = ptx::smem_addr(smem + L.accf_off);
            const uint32_t fv = fk + pa.max_nodes * dk * 2;
            for (int e = lane; e < nacc * (k8 + v8); e += 32) {
                const bool isk = e < nacc * k8;
                const int e2 = isk ? e : e - nacc * k8;
                const int per = isk ? k8 : v8;
                const int node = e2 / per, c8 = (e2 % per) * 8;
                const size_t row = (size_t)(poff + node) * H + h;
                if (isk)
                    ptx::cp_async_16(fk + (node * dk + c8) * 2, pk + row * dk + c8);
                else
                    ptx::cp_async_16(fv + (node * DV + c8) * 2, pv + row * DV + c8);
            }
            if (lane < nacc) gl = pa.g[(size_t)(poff + lane) * H + h];
            // the greedy walk of the previous tree (LLM Primer VI ch. 9 §9.1) finds the
            // path; every block of the request runs it, the head-0 block writes it out.
            // Lane i loads node i's parent and tokens; then the state copies may start.
            int wp = -1, wd = 0, wt = 0;
            if (lane < nacc) {
                wp = pa.parent[poff + lane];
                wd = P.acc_draft[poff + lane];
                wt = P.acc_target[poff + lane];
            }
            const int32_t root = P.acc_root[b];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_issue);
            int *wpar = reinterpret_cast<int *>(smem + L.acc_off);
            int *wdrf = wpar + pa.max_nodes, *wtgt = wdrf + pa.max_nodes;
            int *wpath = wtgt + pa.max_nodes;
            if (lane < nacc) {
                wpar[lane] = wp;
                wdrf[lane] = wd;
                wtgt[lane] = wt;
            }
            const bool wbad = __any_sync(0xffffffffu, lane < nacc && (wp < -1 || wp >= lane));
            __syncwarp();
            int32_t bonus = -1;
            const int Lw = (prange && !wbad)
                               ? warp_greedy_walk_shared(wpar, wdrf, wtgt, nacc, mdp, root, wpath,
                                                         &bonus)
                               : -1;
            __syncwarp();
            if (h == 0) {
                for (int m = lane; m < mdp; m += 32) P.acc_path[(size_t)b * mdp + m] = m < Lw ? wpath[m] : -1;
                if (lane == 0) {
                    P.acc_len[b] = Lw < 0 ? 0 : Lw;
                    P.acc_bonus[b] = Lw < 0 ? -1 : bonus;
                }
            }
            Lq = Lw < 0 ? 0 : Lw;
            pm = lane < Lq ? wpath[lane] : -1;
            pbad = Lw < 0;
        } else {
            Lq = pa.len[b];
            pm = lane < mdp ? pa.path[(size_t)b * mdp + lane] : -1;
            pbad = !prange || Lq < 0 || Lq > mdp;
            pbad = pbad || __any_sync(0xffffffffu, lane < Lq && (pm < 0 || pm >= pn));
        }
        // one round trip: the path's parents and decays, and its factor rows (16-byte
        // copies into shared memory, scaled once the decays are known).  In accept mode
        // they are already requested, and the walk's path is a root path by construction.
        int ppar = -2;
        float pg = 0.f;
        const uint32_t dk16 = ptx::smem_addr(smem + L.pk16_off);
        const uint32_t dv16 = ptx::smem_addr(smem + L.pv16_off);
        if (P.acc) {
            const float gp = __shfl_sync(0xffffffffu, gl, lane < Lq ? pm & 31 : 0);
            if (lane < Lq) pg = gp;
        } else if (!pbad) {
            if (lane < Lq) {
                ppar = pa.parent[poff + pm];
                pg = pa.g[(size_t)(poff + pm) * H + h];
            }
            const int items = Lq * (k8 + v8);
            for (int base = 0; base < items; base += 32) {
                const int e = base + lane;
                const bool isk = e < Lq * k8;
                const int e2 = isk ? e : e - Lq * k8;
                const int per = isk ? k8 : v8;
                const int m = e < items ? e2 / per : 0;
                const int node = __shfl_sync(0xffffffffu, pm, m);
                if (e < items) {
                    const int c8 = (e2 % per) * 8;
                    const size_t row = (size_t)(poff + node) * H + h;
                    if (isk)
                        ptx::cp_async_16(dk16 + (m * dk + c8) * 2, pk + row * dk + c8);
                    else
                        ptx::cp_async_16(dv16 + (m * DV + c8) * 2, pv + row * DV + c8);
                }
            }
        }
        if (!P.acc) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_issue);  // the path's loads are out
        }
        if (!pbad && !P.acc) {
            const int prev = __shfl_up_sync(0xffffffffu, pm, 1);
            pbad = __any_sync(0xffffffffu, lane < Lq && ppar != (lane == 0 ? -1 : prev));
        }
        const int Lp = pbad ? 0 : Lq;
        // suffix sums of g along the path, added from the path's end as the commit
        // kernel does (so both give the same bits)
        const float gm = lane < Lp ? pg : 0.f;
        float suf = 0.f, total = 0.f;
        for (int mm = Lp - 1; mm >= 0; --mm) {
            const float y = __shfl_sync(0xffffffffu, gm, mm);
            if (mm > lane) suf += y;
            total += y;
        }
        const float scale = expf(suf);
        ptx::cp_async_wait_all();
        __syncwarp();
        // factor rows: a_m = e^{G_L - G_{p_m}} k_{p_m} and v_{p_m}, fp32
        float *sPA = reinterpret_cast<float *>(smem + L.pa_off);
        float *sPV = reinterpret_cast<float *>(smem + L.pvv_off);
        // the staged rows: by path slot, or in accept mode by node
        const __nv_bfloat16 *k16 = reinterpret_cast<const __nv_bfloat16 *>(
            smem + (P.acc ? L.accf_off : L.pk16_off));
        const __nv_bfloat16 *v16 =
            P.acc ? k16 + pa.max_nodes * dk
                  : reinterpret_cast<const __nv_bfloat16 *>(smem + L.pv16_off);
        const int items = Lp * (k8 + v8);
        for (int base = 0; base < items; base += 32) {
            const int e = base + lane;
            const bool isk = e < Lp * k8;
            const int e2 = isk ? e : e - Lp * k8;
            const int per = isk ? k8 : v8;
            const int m = e < items ? e2 / per : 0;
            const float sc = __shfl_sync(0xffffffffu, scale, m);
            const int srow = P.acc ? __shfl_sync(0xffffffffu, pm, m) : m;
            if (e < items) {
                const int c8 = (e2 % per) * 8;
                const uint4 raw = *reinterpret_cast<const uint4 *>(isk ? k16 + srow * dk + c8
                                                                       : v16 + srow * DV + c8);
                const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                float *dst = isk ? sPA + m * dk + c8 : sPV + m * DV + c8;
                const float f = isk ? sc : 1.f;
                float4 lo4, hi4;
                lo4.x = __low2float(x2[0]) * f; lo4.y = __high2float(x2[0]) * f;
                lo4.z = __low2float(x2[1]) * f; lo4.w = __high2float(x2[1]) * f;
                hi4.x = __low2float(x2[2]) * f; hi4.y = __high2float(x2[2]) * f;
                hi4.z = __low2float(x2[3]) * f; hi4.w = __high2float(x2[3]) * f;
                *reinterpret_cast<float4 *>(dst) = lo4;
                *reinterpret_cast<float4 *>(dst + 4) = hi4;
            }
        }
        if (lane == 0) {
            if (pbad && h == 0) report(a.status, TV_ERR_TREE);
            meta[kMetaPL] = Lp;
            meta[kMetaAlpha] = __float_as_int(expf(total));
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_pend);
    } else if (warp == 7 && lane == 0) {
        // ================= products (one thread)
        bool ok = ptx::mbar_wait(b_qkv, 0, kWaitLimit);
        int n = 0;
        if (ok) {
            int off0 = 0;
            if (!request_range(a.node_offsets, b, a.T, a.max_nodes, off0, n)) n = 0;
        } else {
            atomicOr(sLate, 16);
        }
        const uint32_t idn = (ptx::idesc_bf16_f32(128, 16) & ~(0x3Fu << 17)) |
                             (static_cast<uint32_t>(((n + 15) & ~15) >> 3) << 17);
        if (ok && n > 0) {
            ptx::tc_fence_after_sync();
            // D_S = Q K^T: A = the q tile (M = 128 rows from its start), B = the k tile
            const uint32_t qa = ptx::smem_addr(smem + L.q_off);
            const uint32_t ka = ptx::smem_addr(smem + L.k_off);
            for (int kk = 0; kk < dk / 16; ++kk) {
                const uint32_t o = (kk / 4) * tile_slab + (kk % 4) * 32;
                ptx::mma_bf16(tmem + kColT, ptx::desc_kmajor_sw128(qa + o, 1024),
                              ptx::desc_kmajor_sw128(ka + o, 1024), idn, kk > 0 ? 1u : 0u);
            }
        }
        ptx::mma_commit(b_sfull);
        // context products, chunk by chunk as each is rewritten (A MN-major)
        for (int c = 0; c < nch && ok; ++c) {
            if (!ptx::mbar_wait(b_conv(c), 0, kWaitLimit)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            if (n == 0) continue;
            const uint32_t qa = ptx::smem_addr(smem + L.q_off);
            const uint32_t ca = ptx::smem_addr(sH) + c * kChunkBytes;
            if constexpr (kStateTmem) {
#pragma unroll
                for (int ks = 0; ks < R / 16; ++ks) {
                    const int kk = (c * R) / 16 + ks;  // 16-row step of the key channels
                    const uint64_t bd =
                        ptx::desc_kmajor_sw128(qa + (kk / 4) * tile_slab + (kk % 4) * 32, 1024);
                    // A = the hi (lanes 0-63) and lo (64-127) parts in tensor memory
                    ptx::mma_bf16_ts(tmem, tmem + kColA + c * (R / 2) + ks * 8, bd, idn,
                                     (c > 0 || ks > 0) ? 1u : 0u);
                }
                continue;
            }
#pragma unroll
            for (int g = 0; g < MG; ++g)
#pragma unroll
                for (int ks = 0; ks < R / 16; ++ks) {
                    const int kk = (c * R) / 16 + ks;  // 16-row step of the key channels
                    const uint64_t bd =
                        ptx::desc_kmajor_sw128(qa + (kk / 4) * tile_slab + (kk % 4) * 32, 1024);
                    // rows 0-63: hi block, rows 64-127: lo block
                    const uint64_t ad =
                        ptx::desc_mnmajor_sw128(ca + g * (2 * R * 128) + ks * 2048, R * 128, 1024);
                    ptx::mma_bf16(tmem + g * NP, ad, bd, idn | (1u << 15),
                                  (c > 0 || ks > 0) ? 1u : 0u);
                }
        }
        if (ok && !ptx::mbar_wait(b_wready, 0, kWaitLimit)) ok = false;
        if (ok) {
            ptx::tc_fence_after_sync();
            if (meta[kMetaRun]) {
                // D_T = V^T W^T: A = the v block of a channel group (rows 64-127 are
                // never read), B = W hi, then W lo
                const int npad = (n + 15) & ~15;
                const uint32_t va = ptx::smem_addr(smem + L.v_off);
                const uint32_t wh = ptx::smem_addr(smem + L.whi_off);
                const uint32_t wl = ptx::smem_addr(smem + L.wlo_off);
                constexpr uint32_t kSboW = (NP / 8) * 128;
#pragma unroll
                for (int g = 0; g < MG; ++g)
                    for (int ks = 0; ks < npad / 16; ++ks) {
                        const uint64_t ad =
                            ptx::desc_mnmajor_sw128(va + g * tile_slab + ks * 2048u, tile_slab, 1024);
                        ptx::mma_bf16(tmem + kColT + g * NP, ad,
                                      ptx::desc_kmajor_noswizzle(wh + ks * 256u, 128, kSboW),
                                      idn | (1u << 15), ks > 0 ? 1u : 0u);
                        ptx::mma_bf16(tmem + kColT + g * NP, ad,
                                      ptx::desc_kmajor_noswizzle(wl + ks * 256u, 128, kSboW),
                                      idn | (1u << 15), 1u);
                    }
            }
        }
        if (!ok) atomicOr(sLate, 32);
        ptx::mma_commit(b_dfull);
        // products in flight complete before the epilogue or the exit reads on
        if (!ptx::mbar_wait(b_dfull, 0, kWaitLimit)) atomicOr(sLate, 64);
        meta[kMetaHave] = ok ? 1 : 0;
    }

    // ================= join, then the epilogue (all warps)
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const int late = *sLate;
    const int n = meta[kMetaN], off = meta[kMetaOff];
    const bool run = meta[kMetaRun] != 0 && meta[kMetaHave] != 0 && late == 0;
    if (tid == 0 && late) report(a.status, TV_ERR_TIMEOUT);
    if (meta[kMetaZero])
        for (int e = tid; e < n * DV; e += kThreadsF)
            a.out[((size_t)(off + e / DV) * H + h) * DV + e % DV] = 0.f;
    if (run) {
        // warp w: lane quadrant w % 4 of the accumulators, node half w / 4
        constexpr int HALF = NP / 2;
        const int qd = warp & 3, hf = warp >> 2;
        const int c = 32 * (qd & 1) + lane;  // channel within the 64-channel group
        float *xr = reinterpret_cast<float *>(sH);  // [NP][64], the state is consumed
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * qd) << 16) + hf * HALF;
#pragma unroll
        for (int g = 0; g < MG; ++g) {
            uint32_t cv[HALF], tv[HALF];
            tmem_ld_cols<HALF>(tq + g * NP, cv);
            if (qd < 2) tmem_ld_cols<HALF>(tq + kColT + g * NP, tv);
            ptx::tmem_wait_ld();
            if (qd >= 2)
#pragma unroll
                for (int i = 0; i < HALF; ++i) xr[(hf * HALF + i) * 64 + c] = __uint_as_float(cv[i]);
            __syncthreads();
            if (qd < 2) {
                float *o = a.out + ((size_t)(off + hf * HALF) * H + h) * DV + 64 * g + c;
#pragma unroll
                for (int i = 0; i < HALF; ++i)
                    if (hf * HALF + i < n)
                        o[(size_t)i * H * DV] = sEG[hf * HALF + i] * (__uint_as_float(cv[i]) +
                                                                      xr[(hf * HALF + i) * 64 + c]) +
                                                __uint_as_float(tv[i]);
            }
            __syncthreads();  // the exchange rows are reused by the next group
        }
    }

    // copies still in flight after a failed wait land before the CTA's memory goes away
    if (tid == 0 && late) {
        for (int c = 0; c < nch; ++c) ptx::mbar_wait(b_chunk(c), 0, kWaitLimit);
        ptx::mbar_wait(b_qkv, 0, kWaitLimit);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 7) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// ---------------------------------------------------------------- host side

size_t fused_smem_bytes(const VerifyArgs &a, int pd, int an = 0) {
    const int np = a.max_nodes > 16 ? 32 : 16;
    return FusedLayout(a.dk, a.dv, np, pd, an).total;
}

bool fused_shape_ok(const VerifyArgs &a) {
    return a.decay == TV_DECAY_SCALAR && a.qkv_dtype == TV_BF16 && (a.dk == 64 || a.dk == 128) &&
           (a.dv == 64 || a.dv == 128) && a.max_nodes <= 32 && encode_fn() != nullptr;
}

template <int DV, int NP, bool PEND>
cudaError_t launch_fused_t(const VerifyArgs &a, const PendingArgs *pend, float *Hw, bool expire,
                           cudaStream_t s, const AcceptArgs *acc) {
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv_;
    // q and k: K-major operand tiles; v: MN-major blocks of 64 channels
    if (!(encode_rows(&tq, a.q, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tk, a.k, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tv_, a.v, BF, 2, DV, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B)))
        return cudaErrorInvalidValue;
    FusedParams P;
    P.a = a;
    P.pend = pend ? *pend : PendingArgs{};
    P.H_w = Hw;
    P.wb32 = (reinterpret_cast<uintptr_t>(Hw) & 31u) == 0 ? 1 : 0;
    P.acc = acc != nullptr;
    P.acc_draft = acc ? acc->draft : nullptr;
    P.acc_target = acc ? acc->target : nullptr;
    P.acc_root = acc ? acc->root : nullptr;
    P.acc_len = acc ? acc->len : nullptr;
    P.acc_path = acc ? acc->path : nullptr;
    P.acc_bonus = acc ? acc->bonus : nullptr;
    P.tmem_cols = tmem_columns(2 * (DV / 64) * NP + (DV == 64 && !PEND ? a.dk / 2 : 0));
    P.expire_first_wait = expire ? 1 : 0;
    auto kern = verify_tc_fused_kernel<DV, NP, PEND>;
    cudaError_t e = configure_smem_once(kern, true);
    if (e != cudaSuccess) return e;
    const size_t smem = fused_smem_bytes(a, PEND ? pend->max_depth : 0,
                                         PEND && acc ? pend->max_nodes : 0);
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = resident_ctas(kern, kThreadsF, smem, P.tmem_cols, per_sm)) != cudaSuccess)
        return e;
    P.wave = sms * per_sm;
    return launch_pdl(kern, dim3((unsigned)(a.B * a.H)), dim3(kThreadsF), smem, s, tq, tk, tv_, P);
}

template <bool PEND>
cudaError_t launch_fused(const VerifyArgs &a, const PendingArgs *pend, float *Hw, bool expire,
                         cudaStream_t s, const AcceptArgs *acc = nullptr) {
    const bool np16 = a.max_nodes <= 16;
    if (a.dv == 64)
        return np16 ? launch_fused_t<64, 16, PEND>(a, pend, Hw, expire, s, acc)
                    : launch_fused_t<64, 32, PEND>(a, pend, Hw, expire, s, acc);
    return np16 ? launch_fused_t<128, 16, PEND>(a, pend, Hw, expire, s, acc)
                : launch_fused_t<128, 32, PEND>(a, pend, Hw, expire, s, acc);
}

}  // namespace

bool verify_tc_fused_supported(const VerifyArgs &a) {
    return fused_shape_ok(a) && fused_smem_bytes(a, 0) <= kSmemLimit;
}

bool commit_verify_fused_supported(const VerifyArgs &a, const PendingArgs &p) {
    return fused_shape_ok(a) && fused_smem_bytes(a, p.max_depth) <= kSmemLimit;
}

cudaError_t launch_verify_tc_fused(const VerifyArgs &a, cudaStream_t s, bool expire_first_wait) {
    if (!verify_tc_fused_supported(a)) return cudaErrorNotSupported;
    return launch_fused<false>(a, nullptr, nullptr, expire_first_wait, s);
}

cudaError_t launch_commit_verify_fused(const VerifyArgs &a, const PendingArgs &p, float *H,
                                       cudaStream_t s) {
    if (!commit_verify_fused_supported(a, p)) return cudaErrorNotSupported;
    return launch_fused<true>(a, &p, H, false, s);
}

bool accept_commit_verify_fused_supported(const VerifyArgs &a, const PendingArgs &p) {
    // the previous tree's nodes' factor rows are staged whole (one per lane's decay)
    return fused_shape_ok(a) && p.max_nodes <= 32 &&
           fused_smem_bytes(a, p.max_depth, p.max_nodes) <= kSmemLimit;
}

cudaError_t launch_accept_commit_verify_fused(const VerifyArgs &a, const PendingArgs &p,
                                              const AcceptArgs &acc, float *H, cudaStream_t s) {
    if (!accept_commit_verify_fused_supported(a, p)) return cudaErrorNotSupported;
    return launch_fused<true>(a, &p, H, false, s, &acc);
}

}  // namespace tv
