// tree_attention.cu -- tree-masked softmax attention over a shared-prefix KV cache:
// the attention layers' share of verifying a draft tree in a hybrid model.
//
// LLM Primer VI ch. 9: the target runs one forward pass over the prefix followed by
// the candidates (§9.1), and a candidate tree is verified in one attention pass with
// a custom mask (§9.2).  Bole summary page ("Why existing tree speculation fails on
// hybrid models"): every branch shares the prefix's KV and adds only its own.  So
// query row (node i, head h) of request b attends to the first ctx_len[b] cached
// positions of KV head h / (H / Hkv) and to the tree nodes on i's root path, i
// included:  o = sum_j softmax_j(scale * q . k_j) v_j.
//
// Work unit: (request b, KV head, M tile of 128 query rows, split of the context).
// Row r of an M tile is (node mt * 128 / grp + r / grp, head kvh * grp + r % grp), so
// the grp query heads of a KV head share every key tile.  Keys come in tiles of 128:
// the split's context tiles, then (split 0 only) the request's tree nodes under the
// ancestor mask.  Warp roles: warp 0 issues TMA copies (lane 0: Q once, then K tiles;
// lane 1: V tiles; each into its own ring), warp 1 issues tcgen05 MMAs, warps 2-5 own
// one query row per thread.  Per tile:
//   S = Q K^T        tcgen05 kind::f16, M = 128, N = 128 keys, K = d, into one of two
//                    tensor-memory S/P buffers (S of the next tile is formed while the
//                    softmax works on this one);
//   P = 2^(S * scale * log2 e - m) in fp32, split into bf16 hi (upper 16 bits) and
//                    lo = bf16(P - hi) parts (|P - hi - lo| <= 2^-16 P), written by the
//                    softmax threads over the same buffer (two keys per column, hi in
//                    columns 0-63, lo in 64-127);
//   O += P V         A = P hi, then P lo, from tensor memory, M = 128, N = d, K = 128
//                    keys, with V read as an MN-major operand straight from its TMA
//                    tile; O stays in tensor memory.  The row sums l of the fp32
//                    weights are kept by the softmax threads in registers.
// The MMA thread issues whichever of the next S and the next P V is ready, so a K tile
// still in flight never holds back P V, and a buffer takes the next S only after its
// P V is done.  The reference maximum m of a row is raised only when a tile's maximum
// exceeds it by more than 8 (log2 units); O and l are then rescaled in tensor memory
// before the tile's P V, so P <= 2^8 always.  Context positions at or beyond ctx_len,
// and tree nodes off the row's root path, get weight 0, and the V rows of such keys
// are zeroed in shared memory before P V, so whatever the cache holds there never
// reaches O.  A warp whose 32 rows are all padding (rows past the request's last
// query) only takes part in the handshakes.
//
// With one split the epilogue writes O / l.  With several, each split writes
// (O, m, l) per row to the caller's workspace and a second kernel merges them.
// Every mbarrier wait is bounded: on expiry the CTA records TV_ERR_TIMEOUT, its roles
// stop, in-flight copies and MMAs are waited for, and tensor memory is freed.
#include <algorithm>

#include "tc_common.cuh"

namespace tv {
namespace {

using tcc::kWaitLimit;

constexpr int kThreadsAt = 192;
constexpr uint32_t kSlab = 128 * 128;  // 128 rows x 128 bytes (64 bf16), swizzled
constexpr float kHeadroom = 8.f;       // log2 units of growth before a rescale
constexpr uint32_t kTmemCols = 512;    // S/P buffers at 0 and 128, O at 256

// Shared memory: Q, a ring of KS K tiles and one of VS V tiles (128 keys each).
// At d = 128 both rings are 3 deep (224 KB of tiles), at d = 64 both are 6 deep.
template <int D>
struct AttnLayout {
    static constexpr int KS = D == 128 ? 3 : 6;
    static constexpr int VS = D == 128 ? 3 : 6;
    static constexpr uint32_t kAtoms = D / 64;          // 64-element slabs of a row
    static constexpr uint32_t kHalf = kAtoms * kSlab;   // one K or V tile, one Q tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kHalf;           // K tiles [KS]
    static constexpr uint32_t kV = kK + KS * kHalf;      // V tiles [VS]
    static constexpr uint32_t kPar = kV + VS * kHalf;  // parent [kMaxNodes] int16
    static constexpr uint32_t kBar = kPar + kMaxNodes * 2;
    // mbarrier slots: Q landed; K, V tiles landed / free; per tensor-memory S/P
    // buffer: S ready, S read, P written, P V done; every MMA done
    static constexpr int kQBar = 0, kKFull = 1, kVFull = kKFull + KS, kKFree = kVFull + VS,
                         kVFree = kKFree + KS, kSBar = kVFree + VS, kSFree = kSBar + 2,
                         kPBar = kSFree + 2, kOBar = kPBar + 2, kDone = kOBar + 2,
                         kNumBars = kDone + 1;
    static constexpr uint32_t kMisc = kBar + kNumBars * 8;  // tmem slot, flags
    static constexpr uint32_t kBytes = kMisc + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;       // base alignment slack
};

struct AttnParams {
    AttnArgs a;
    int grp, mts, ns;
    float sl2;  // scale * log2(e)
};

// Wait for a phase, giving up when the CTA's abort flag is raised or the limit passes.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort,
                                           uint32_t suspend_ns = 20000) {
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(bar, parity, suspend_ns)) {
        if (*abort || clock64() - t0 > kWaitLimit) {
            *abort = 1;
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Partial results of a split: O rows first, then (m, l) pairs.
__device__ __forceinline__ float *part_o(const AttnParams &P, size_t u, int r, int D) {
    return P.a.ws + (u * 128 + r) * D;
}
__device__ __forceinline__ float *part_ml(const AttnParams &P, size_t units_all, size_t u, int r,
                                          int D) {
    return P.a.ws + units_all * 128 * D + (u * 128 + r) * 2;
}

template <int D>
__global__ void __launch_bounds__(kThreadsAt, 1)
    tree_attention_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_kc,
                          const __grid_constant__ CUtensorMap tm_vc,
                          const __grid_constant__ CUtensorMap tm_kt,
                          const __grid_constant__ CUtensorMap tm_vt, const AttnParams P) {
    using Lay = AttnLayout<D>;
    constexpr int KS = Lay::KS, VS = Lay::VS;
    constexpr int kQBar = Lay::kQBar, kKFull = Lay::kKFull, kVFull = Lay::kVFull,
                  kKFree = Lay::kKFree, kVFree = Lay::kVFree, kSBar = Lay::kSBar,
                  kSFree = Lay::kSFree, kPBar = Lay::kPBar, kOBar = Lay::kOBar, kDone = Lay::kDone;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const AttnArgs &a = P.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int blk = blockIdx.x;
    const int split = blk % P.ns;
    blk /= P.ns;
    const int mt = blk % P.mts;
    blk /= P.mts;
    const int kvh = blk % a.Hkv;
    const int b = blk / a.Hkv;
    const int grp = P.grp, npt = 128 / grp;
    const bool first_cta = kvh == 0 && mt == 0 && split == 0;

    int16_t *s_par = reinterpret_cast<int16_t *>(sm + Lay::kPar);
    volatile int *s_flags = reinterpret_cast<volatile int *>(sm + Lay::kMisc + 4);  // bad, abort
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + Lay::kMisc);
    const uint32_t sbase = ptx::smem_addr(sm);
    auto bar = [&](int i) { return sbase + Lay::kBar + 8u * (uint32_t)i; };

    // ---- set-up that reads nothing an earlier kernel writes: it overlaps that
    // kernel's tail (programmatic dependent launch)
    if (tid == 0) {
        s_flags[0] = 0;
        s_flags[1] = 0;
        for (int i = 0; i < Lay::kNumBars; ++i) {
            // arrived on by the 128 softmax threads
            const bool all = i == kPBar || i == kPBar + 1 || i == kSFree || i == kSFree + 1;
            ptx::mbar_init(bar(i), all ? 128u : 1u);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_kc);
        ptx::prefetch_tensormap(&tm_vc);
        ptx::prefetch_tensormap(&tm_kt);
        ptx::prefetch_tensormap(&tm_vt);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(s_tmem), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    volatile int *abort = s_flags + 1;

    pdl_wait();
    pdl_launch_next();

    // ---- this CTA's rows and key tiles
    int off = 0, n = 0;
    const bool range = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    const int nrows = range ? min(n * grp - mt * 128, 128) : 0;
    const int L = a.ctx_len[b];  // read alongside the offsets (b < B always)
    const bool ctx_ok = !range || (L >= 0 && L <= a.P);
    const int ct = ctx_ok ? (L + 127) / 128 : 0;
    const int c0 = (int)((long long)ct * split / P.ns);
    const int c1 = (int)((long long)ct * (split + 1) / P.ns);
    const int nctx = c1 - c0;
    const int nt = nctx + (split == 0 ? (n + 127) / 128 : 0);
    const size_t units_all = (size_t)a.B * a.Hkv * P.mts * P.ns;
    const size_t unit = (((size_t)b * a.Hkv + kvh) * P.mts + mt) * P.ns + split;
    if (tid == 0 && first_cta && !range) report(a.status, TV_ERR_TREE);
    if (tid == 0 && first_cta && range && !ctx_ok) report(a.status, TV_ERR_SHAPE);
    // run the pipeline, or only write the rows' empty results, or nothing at all
    const bool run = nrows > 0 && ctx_ok && nt > 0;
    const bool empty_rows = nrows > 0 && !run;

    // rows without a result (malformed input, or a split with no keys)
    auto write_empty = [&](int t0, int nthreads) {
        for (int e = t0; e < nrows * D; e += nthreads) {
            const int r = e / D, c = e % D;
            const int row = mt * 128 + r;
            if (P.ns == 1) {
                const size_t node = (size_t)off + row / grp;
                a.out[(node * a.H + kvh * grp + row % grp) * D + c] = 0.f;
            } else {
                part_o(P, unit, r, D)[c] = 0.f;
                if (c == 0) {
                    part_ml(P, units_all, unit, r, D)[0] = neg_inf();
                    part_ml(P, units_all, unit, r, D)[1] = 0.f;
                }
            }
        }
    };
    if (empty_rows) write_empty(tid, kThreadsAt);

    const uint32_t sQ = sbase + Lay::kQ;
    auto sK = [&](int s) { return sbase + Lay::kK + (uint32_t)s * Lay::kHalf; };
    auto sV = [&](int s) { return sbase + Lay::kV + (uint32_t)s * Lay::kHalf; };
    // ring slot of tile j and the parity of its use of that slot
    auto kslot = [](int j) { return j % KS; };
    auto kpar = [](int j) { return (uint32_t)((j / KS) & 1); };
    auto vslot = [](int j) { return j % VS; };
    auto vpar = [](int j) { return (uint32_t)((j / VS) & 1); };
    constexpr uint32_t kOCol = 256;

    if (!run) {
        // nothing to compute
    } else if (warp == 0) {
        // ------------------------------------------------ TMA producers: lane 0 Q and K
        // tiles, lane 1 V tiles, each with its own ring
        if (lane < 2) {
            const bool is_k = lane == 0;
            const int depth = is_k ? KS : VS;
            const CUtensorMap *mc = is_k ? &tm_kc : &tm_vc;
            const CUtensorMap *mtree = is_k ? &tm_kt : &tm_vt;
            const int full0 = is_k ? kKFull : kVFull, free0 = is_k ? kKFree : kVFree;
            if (is_k) {
                ptx::mbar_arrive_expect_tx(bar(kQBar), Lay::kHalf);
                for (int at = 0; at < (int)Lay::kAtoms; ++at)
                    ptx::tma_load_4d(sQ + at * kSlab, &tm_q, 64 * at, 0, kvh, off + mt * npt,
                                     bar(kQBar));
            }
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int s = j % depth;
                if (j >= depth && !wait_phase(bar(free0 + s), ((j / depth) - 1) & 1, abort)) break;
                const uint32_t dst = is_k ? sK(s) : sV(s);
                ptx::mbar_arrive_expect_tx(bar(full0 + s), Lay::kHalf);
                for (int at = 0; at < (int)Lay::kAtoms; ++at) {
                    if (j < nctx)
                        ptx::tma_load_3d(dst + at * kSlab, mc, 64 * at, 128 * (c0 + j),
                                         b * a.Hkv + kvh, bar(full0 + s));
                    else
                        ptx::tma_load_3d(dst + at * kSlab, mtree, 64 * at, kvh,
                                         off + 128 * (j - nctx), bar(full0 + s));
                }
                issued = j + 1;
            }
            // no copy may still be landing when the CTA ends
            if (is_k) ptx::mbar_wait(bar(kQBar), 0, kWaitLimit);
            for (int j = max(0, issued - depth); j < issued; ++j)
                ptx::mbar_wait(bar(full0 + j % depth), (j / depth) & 1, kWaitLimit);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer: S = Q K^T into an
        // S/P buffer as soon as a K tile is in and the buffer's previous P V is done;
        // P V (and the row sums P 1) as soon as P is written; neither waits for the other
        if (lane == 0) {
            constexpr uint32_t idS = ptx::idesc_bf16_f32(128, 128);
            constexpr uint32_t idPV = ptx::idesc_bf16_f32_bmn(128, D);
            bool ok = wait_phase(bar(kQBar), 0, abort);
            int js = 0, jp = 0;
            long long t_last = clock64();
            while (ok && jp < nt) {
                bool progressed = false;
                if (js < nt && ptx::mbar_test_wait(bar(kKFull + kslot(js)), kpar(js)) &&
                    (js < 2 ||
                     (ptx::mbar_test_wait(bar(kSFree + (js & 1)), ((js >> 1) - 1) & 1) &&
                      ptx::mbar_test_wait(bar(kOBar + (js & 1)), ((js >> 1) - 1) & 1)))) {
                    const int s = js & 1, ks = kslot(js);
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = (kk >> 2) * kSlab + (kk & 3) * 32;
                        ptx::mma_bf16(tmem + 128u * s, ptx::desc_kmajor_sw128(sQ + o, 1024),
                                      ptx::desc_kmajor_sw128(sK(ks) + o, 1024), idS, kk > 0);
                    }
                    ptx::mma_commit(bar(kSBar + s));
                    ptx::mma_commit(bar(kKFree + ks));
                    ++js;
                    progressed = true;
                }
                if (jp < js && ptx::mbar_test_wait(bar(kPBar + (jp & 1)), (jp >> 1) & 1) &&
                    ptx::mbar_test_wait(bar(kVFull + vslot(jp)), vpar(jp))) {
                    const int s = jp & 1, vs = vslot(jp);
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // P: 16 keys = 8 columns of packed bf16 pairs per step, the hi
                        // part at column 8 kk, the lo part 64 columns further
                        const uint32_t pa = tmem + 128u * s + 8u * kk;
                        const uint64_t bd = ptx::desc_mnmajor_sw128(sV(vs) + kk * 2048u,
                                                                    D == 128 ? kSlab : 0u, 1024);
                        const uint32_t acc = (jp > 0 || kk > 0) ? 1u : 0u;
                        ptx::mma_bf16_ts(tmem + kOCol, pa, bd, idPV, acc);
                        ptx::mma_bf16_ts(tmem + kOCol, pa + 64u, bd, idPV, 1u);
                    }
                    ptx::mma_commit(bar(kOBar + s));
                    ptx::mma_commit(bar(kVFree + vs));
                    ++jp;
                    progressed = true;
                }
                if (progressed) {
                    t_last = clock64();
                } else {
                    // sleep on the event most likely next
                    if (jp < js)
                        ptx::mbar_try_wait(bar(kPBar + (jp & 1)), (jp >> 1) & 1, 1000);
                    else
                        ptx::mbar_try_wait(bar(kKFull + kslot(js)), kpar(js), 1000);
                    if (*abort || clock64() - t_last > kWaitLimit) {
                        *abort = 1;
                        ok = false;
                    }
                }
            }
            // every MMA issued has completed before tensor memory is freed
            ptx::mma_commit(bar(kDone));
            ptx::mbar_wait(bar(kDone), 0, kWaitLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax: one query row per thread
        const int quad = warp & 3;
        const int r = 32 * quad + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
        const bool row_valid = r < nrows;
        const bool warp_live = 32 * quad < nrows;  // a warp of padding rows only keeps time
        const int row = mt * 128 + r;
        const int node = row / grp;
        const float sl2 = P.sl2;
        // the tree (parents precede children), checked while the first tiles load
        for (int i = tid - 64; i < n; i += 128) {
            const int p = a.parent[off + i];
            s_par[i] = (int16_t)p;
            if (p < -1 || p >= i) s_flags[0] = 1;
        }
        tcc::named_barrier(1, 128);
        const bool bad = s_flags[0] != 0;
        if (bad && tid == 64 && first_cta) report(a.status, TV_ERR_TREE);
        float m = neg_inf();
        float lsum = 0.f;  // the row's sum of weights, relative to 2^m
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int s = j & 1;
            if (!__all_sync(0xffffffffu, wait_phase(bar(kSBar + s), (j >> 1) & 1, abort))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            float x[128];
            if (warp_live) {
                uint32_t u[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) ptx::tmem_ld_x32_nowait(tl + 128u * s + 32u * c, u[c]);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(u[c][e]);
            }
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(kSFree + s));

            const bool ctx_tile = j < nctx;
            const int vk = ctx_tile ? min(128, L - 128 * (c0 + j)) : min(128, n - 128 * (j - nctx));
            float t = neg_inf();
            if (warp_live) {
                // keys outside the context or off the root path: -inf
                if (ctx_tile && vk < 128) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) x[c] = c < vk ? x[c] : neg_inf();
                } else if (!ctx_tile) {
                    const int tbase = 128 * (j - nctx);
                    uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
                    if (row_valid && !bad) {
                        for (int q = node; q >= 0; q = s_par[q]) {
                            const int rel = q - tbase;
                            if (rel >= 0 && rel < 128) {
                                const uint32_t bit = 1u << (rel & 31);
                                const int w = rel >> 5;
                                w0 |= w == 0 ? bit : 0u;
                                w1 |= w == 1 ? bit : 0u;
                                w2 |= w == 2 ? bit : 0u;
                                w3 |= w == 3 ? bit : 0u;
                            }
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const uint32_t w = c < 32 ? w0 : c < 64 ? w1 : c < 96 ? w2 : w3;
                        x[c] = (w >> (c & 31)) & 1u ? x[c] : neg_inf();
                    }
                }
                float tm[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) tm[e] = x[e];
#pragma unroll
                for (int c = 8; c < 128; c += 8)
#pragma unroll
                    for (int e = 0; e < 8; ++e) tm[e] = fmaxf(tm[e], x[c + e]);
                t = fmaxf(fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])),
                          fmaxf(fmaxf(tm[4], tm[5]), fmaxf(tm[6], tm[7]))) * sl2;
            }

            // raise the reference maximum; O and l are rescaled in tensor memory once
            // the previous tile's P V is done (it is issued only after this arrives)
            const bool need = t > m + kHeadroom;
            if (__any_sync(0xffffffffu, need) && j > 0) {
                if (!__all_sync(0xffffffffu, wait_phase(bar(kOBar + ((j - 1) & 1)),
                                                        ((j - 1) >> 1) & 1, abort, 2000))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const float alpha = need ? (m == neg_inf() ? 0.f : ex2(m - t)) : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld_x32_nowait(tl + kOCol + 32u * c, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    ptx::tmem_st_x32(tl + kOCol + 32u * c, o);
                }
                lsum *= alpha;
            }
            if (need) m = t;

            // P over this tile's S buffer (S is in registers), split into bf16 hi and lo
            // parts: hi keeps the upper 16 bits of each fp32 weight, lo = bf16(p - hi),
            // so p - hi - lo <= 2^-16 p; hi pairs in columns 0-63, lo pairs in 64-127
            if (warp_live) {
                const float nm = m == neg_inf() ? 0.f : -m;
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t ph[16], pl[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = ex2(fmaf(x[32 * q + 2 * e], sl2, nm));
                        const float p1 = ex2(fmaf(x[32 * q + 2 * e + 1], sl2, nm));
                        ls0 += p0;
                        ls1 += p1;
                        tcc::split_pair(p0, p1, ph[e], pl[e]);
                    }
                    ptx::tmem_st_x16(tl + 128u * s + 16u * q, ph);
                    ptx::tmem_st_x16(tl + 128u * s + 64u + 16u * q, pl);
                }
                lsum += ls0 + ls1;
            }
            ptx::tmem_wait_st();
            if (vk < 128) {
                // keys past the end of the context or of the tree: zero their V rows
                if (!__all_sync(0xffffffffu, wait_phase(bar(kVFull + vslot(j)), vpar(j), abort))) {
                    ok = false;
                    break;
                }
                uint8_t *vbase = sm + Lay::kV + (uint32_t)vslot(j) * Lay::kHalf;
                const int per_slab = (128 - vk) * 8;
                for (int e = r; e < per_slab * (int)Lay::kAtoms; e += 128) {
                    const int slab = e / per_slab, rem = e % per_slab;
                    *reinterpret_cast<uint4 *>(vbase + slab * kSlab + (vk + rem / 8) * 128 +
                                               (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(kPBar + s));
        }

        // epilogue
        if (ok && __all_sync(0xffffffffu, wait_phase(bar(kOBar + ((nt - 1) & 1)),
                                                     ((nt - 1) >> 1) & 1, abort))) {
            ptx::tc_fence_after_sync();
            if (warp_live) {
                const float l = bad ? 0.f : lsum;
                if (bad) m = neg_inf();  // a malformed tree: zero rows
                const float inv = l > 0.f ? 1.f / l : 0.f;
                float *dst;
                if (P.ns == 1) {
                    const size_t nd = (size_t)off + (row_valid ? node : 0);
                    dst = a.out + (nd * a.H + kvh * grp + row % grp) * D;
                } else {
                    dst = part_o(P, unit, r, D);
                }
                const float sc = bad ? 0.f : P.ns == 1 ? inv : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld_x32_nowait(tl + kOCol + 32u * c, o);
                    ptx::tmem_wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4 *>(dst + 32 * c + e) =
                                make_float4(__uint_as_float(o[e]) * sc, __uint_as_float(o[e + 1]) * sc,
                                            __uint_as_float(o[e + 2]) * sc,
                                            __uint_as_float(o[e + 3]) * sc);
                    }
                }
                if (P.ns > 1 && row_valid) {
                    part_ml(P, units_all, unit, r, D)[0] = m;
                    part_ml(P, units_all, unit, r, D)[1] = l;
                }
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort) report(a.status, TV_ERR_TIMEOUT);
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge of the splits' partial results, one CTA per query row (one thread per
// channel): out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s with M = max_s m_s.
template <int D>
__global__ void __launch_bounds__(D) tree_attention_merge_kernel(const AttnParams P) {
    __shared__ float s_w[64];
    __shared__ float s_den;
    const AttnArgs &a = P.a;
    const int r = blockIdx.x % 128;
    int blk = blockIdx.x / 128;
    const int mt = blk % P.mts;
    blk /= P.mts;
    const int kvh = blk % a.Hkv, b = blk / a.Hkv;
    const int grp = P.grp, ns = P.ns, c = threadIdx.x;
    pdl_wait();
    pdl_launch_next();
    int off, n;
    if (!request_range(a.node_offsets, b, a.T, a.max_nodes, off, n)) return;
    if (r >= min(n * grp - mt * 128, 128)) return;
    const size_t units_all = (size_t)a.B * a.Hkv * P.mts * ns;
    const size_t u0 = (((size_t)b * a.Hkv + kvh) * P.mts + mt) * ns;
    if (c < 32) {  // splits c and c + 32 (at most 64)
        const float *ml0 = part_ml(P, units_all, u0 + c, r, D);
        const float *ml1 = part_ml(P, units_all, u0 + c + 32, r, D);
        const float m0 = c < ns ? ml0[0] : neg_inf(), l0 = c < ns ? ml0[1] : 0.f;
        const float m1 = c + 32 < ns ? ml1[0] : neg_inf(), l1 = c + 32 < ns ? ml1[1] : 0.f;
        float M = fmaxf(m0, m1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w0 = m0 == neg_inf() ? 0.f : exp2f(m0 - M);
        const float w1 = m1 == neg_inf() ? 0.f : exp2f(m1 - M);
        const float den = warp_sum(w0 * l0 + w1 * l1);
        if (c < ns) s_w[c] = w0;
        if (c + 32 < ns) s_w[c + 32] = w1;
        if (c == 0) s_den = den;
    }
    __syncthreads();
    float num = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float w = s_w[s];
        if (w != 0.f) num += w * part_o(P, u0 + s, r, D)[c];
    }
    const int row = mt * 128 + r;
    const size_t node = (size_t)off + row / grp;
    a.out[(node * a.H + kvh * grp + row % grp) * D + c] = s_den > 0.f ? num / s_den : 0.f;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

int m_tiles(const AttnArgs &a) { return (a.max_nodes * (a.H / a.Hkv) + 127) / 128; }

// Context splits: one when the units alone fill half the SMs, else as many as
// keep all CTAs in one wave (one CTA per SM), at most one per context tile and 64.
int pick_splits(const AttnArgs &a) {
    const long long units = (long long)a.B * a.Hkv * m_tiles(a);
    const int sms = sm_count();
    if (units <= 0 || 2 * units >= sms) return 1;
    const long long want = sms / units;
    const long long ctiles = (a.P + 127) / 128;
    return (int)std::max(1LL, std::min(std::min(want, ctiles), 64LL));
}

size_t split_bytes(const AttnArgs &a, int ns) {
    return (size_t)a.B * a.Hkv * m_tiles(a) * ns * 128 * (a.d + 2) * sizeof(float);
}

bool encode_attn_maps(const AttnArgs &a, CUtensorMap *tq, CUtensorMap *tkc, CUtensorMap *tvc,
                      CUtensorMap *tkt, CUtensorMap *tvt) {
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
    const auto fn = tcc::encode_fn();
    if (!fn) return false;
    const cuuint64_t d = (cuuint64_t)a.d, grp = (cuuint64_t)(a.H / a.Hkv);
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    auto enc = [&](CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                   const cuuint64_t *strides, const cuuint32_t *box) {
        return fn(m, BF, rank, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, SW, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    // q [T][Hkv][grp][d]: one box = 128 / grp nodes x grp heads x 64 channels
    const cuuint64_t qd[4] = {d, grp, (cuuint64_t)a.Hkv, (cuuint64_t)a.T};
    const cuuint64_t qs[3] = {d * 2, grp * d * 2, (cuuint64_t)a.H * d * 2};
    const cuuint32_t qb[4] = {64, (cuuint32_t)grp, 1, (cuuint32_t)(128 / grp)};
    // cache [B * Hkv][P][d]: 128 positions x 64 channels
    const cuuint64_t cd[3] = {d, (cuuint64_t)a.P, (cuuint64_t)a.B * a.Hkv};
    const cuuint64_t cs[2] = {d * 2, (cuuint64_t)a.P * d * 2};
    const cuuint32_t cb[3] = {64, 128, 1};
    // tree [T][Hkv][d]: 128 nodes x 64 channels of one KV head
    const cuuint64_t td[3] = {d, (cuuint64_t)a.Hkv, (cuuint64_t)a.T};
    const cuuint64_t ts[2] = {d * 2, (cuuint64_t)a.Hkv * d * 2};
    const cuuint32_t tb[3] = {64, 1, 128};
    return enc(tq, a.q, 4, qd, qs, qb) && enc(tkc, a.k_cache, 3, cd, cs, cb) &&
           enc(tvc, a.v_cache, 3, cd, cs, cb) && enc(tkt, a.k_tree, 3, td, ts, tb) &&
           enc(tvt, a.v_tree, 3, td, ts, tb);
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, cudaStream_t s) {
    using Lay = AttnLayout<D>;
    static_assert(Lay::kAlloc <= tcc::kSmemLimit, "shared-memory plan exceeds the limit");
    CUtensorMap tq, tkc, tvc, tkt, tvt;
    if (!encode_attn_maps(a, &tq, &tkc, &tvc, &tkt, &tvt)) return cudaErrorInvalidValue;
    AttnParams P;
    P.a = a;
    P.grp = a.H / a.Hkv;
    P.mts = m_tiles(a);
    P.ns = pick_splits(a);
    if (P.ns > 1 && (!a.ws || a.ws_bytes < split_bytes(a, P.ns))) {
        const size_t per = split_bytes(a, 1);
        const int fit = a.ws ? (int)std::min<size_t>(a.ws_bytes / per, (size_t)P.ns) : 0;
        P.ns = fit >= 2 ? fit : 1;
    }
    P.sl2 = a.scale * 1.4426950408889634f;
    const cudaError_t attr = configure_smem_once(tree_attention_kernel<D>, false);
    if (attr != cudaSuccess) return attr;
    const unsigned grid = (unsigned)((size_t)a.B * a.Hkv * P.mts * P.ns);
    cudaError_t e = launch_pdl(tree_attention_kernel<D>, dim3(grid), dim3(kThreadsAt),
                               (size_t)Lay::kAlloc, s, tq, tkc, tvc, tkt, tvt, P);
    if (e != cudaSuccess || P.ns == 1) return e;
    return launch_pdl(tree_attention_merge_kernel<D>,
                      dim3((unsigned)((size_t)a.B * a.Hkv * P.mts * 128)), dim3(D), 0, s, P);
}

}  // namespace

size_t tree_attention_workspace_bytes(const AttnArgs &a) {
    const int ns = pick_splits(a);
    return ns > 1 ? split_bytes(a, ns) : 0;
}

cudaError_t launch_tree_attention(const AttnArgs &a, cudaStream_t s) {
    if (a.d == 64) return launch_d<64>(a, s);
    if (a.d == 128) return launch_d<128>(a, s);
    return cudaErrorNotSupported;
}

}  // namespace tv
