// verify_tc.cu -- tree verification with the context term on tcgen05 tensor cores.
//
// Tree closed form (Bole summary page, "Core techniques" §1), scalar decay:
//   o_i = e^{G_i} (H0^T q_i) + sum_{j in anc*(i)} e^{G_i - G_j} (q_i . k_j) v_j
// with anc*(i) the root path of node i including i and G_i = sum_{j in anc*(i)} g_j.
// Only the per-token factors are read (§2); no per-node state is formed.
//
// One CTA = one (request, head), 256 threads:
//   * thread 0 issues one bulk copy of the unit's H0 (dk x dv fp32, contiguous)
//     and TMA tensor copies of the request's q rows (128-byte swizzled tiles, the
//     K-major operand layout of the tensor core), all completing on one mbarrier;
//   * meanwhile the warps validate the tree and compute, for every node i and
//     ancestor j, the decayed score w_ij = e^{G_i - G_j} (q_i . k_j) and e^{G_i};
//   * H0 is split in place into bf16 hi + lo parts (H0 = hi + lo + O(2^-17 |H0|))
//     and rewritten transposed as the K-major A operand (rows = value channels);
//   * one thread issues D[c][i] = sum_r A[c][r] q_i[r] on tcgen05 (kind::f16,
//     M = 128, N = nodes rounded up to 16, fp32 accumulators in tensor memory).
//     q is bf16, so hi and lo products are exact and D carries H0^T q to fp32
//     accuracy.  For dv = 64 the hi and lo halves are stacked into one 128-row
//     operand and summed in the epilogue; for dv = 128 they accumulate in place;
//   * the epilogue reads D from tensor memory (lane = value channel), applies
//     e^{G_i}, adds sum_j w_ij v_j and stores fp32 rows, 128 bytes per warp.
// Every wait is bounded (TV_ERR_TIMEOUT); malformed trees zero their rows and
// set TV_ERR_TREE.
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kThreads = 256;
// Shared-memory plan, identical on host and device.  TMA destinations and
// 128-byte-swizzled operands are 1024-byte aligned.
//   A region: H0 streams in as kChunkRows-row fp32 chunks; each chunk is split in
//     place into bf16 hi/lo K-major operand rows (value channels) of the same size.
//   scalar decay: q arrives swizzled and is the B operand itself; g is gathered.
//   diagonal decay: q arrives as dense rows; B = bf16 hi/lo of e^{G_i} * q_i is
//     written by the warps in the swizzled layout; g arrives as dense fp32 rows and
//     becomes exp(g) in place.
//   The lo-part exchange (dv = 64) reuses the A region when it is large enough.
//   pending commit (pend_depth > 0): the previous step's path factors, k rows
//     scaled by their suffix decays and v rows, both fp32, plus the path itself.
struct TcLayout {
    uint32_t a_off, b_off, blo_off, q_off, k_off, v_off, e_off, x_off, w_off, anc_off, eg_off,
        g_off, par_off, dep_off, poff_off, pnode_off, bar_off, misc_off, pk_off, pv_off, pg_off,
        ppath_off, pmisc_off, total;
    __host__ __device__ TcLayout(int dk, int dv, int npad_max, int max_depth, bool diag,
                                 int pend_depth = 0) {
        const uint32_t swz_tile = (dk / 64) * npad_max * 128;  // one swizzled [n][dk] bf16 tile
        const uint32_t a_bytes = dk * dv * 4;
        // dv = 64: the epilogue dumps both 64-row halves of D, npad x 128 fp32
        const uint32_t x_bytes = dv == 64 ? npad_max * 128 * 4 : 0;
        const bool x_in_a = x_bytes <= a_bytes;
        a_off = 0;
        b_off = align_up(a_off + a_bytes, 1024);               // B (hi) operand
        blo_off = align_up(b_off + swz_tile, 1024);            // B lo operand (diag)
        q_off = align_up(blo_off + (diag ? swz_tile : 0), 1024);  // dense q rows (diag)
        k_off = align_up(q_off + (diag ? npad_max * dk * 2 : 0), 1024);
        v_off = align_up(k_off + npad_max * dk * 2, 1024);
        e_off = align_up(v_off + npad_max * dv * 2, 1024);      // g -> exp(g) rows (diag)
        x_off = align_up(e_off + (diag ? npad_max * dk * 4 : 0), 16);
        w_off = align_up(x_off + (x_in_a ? 0 : x_bytes), 16);
        if (x_in_a) x_off = a_off;
        anc_off = align_up(w_off + npad_max * max_depth * 4, 16);   // root paths
        eg_off = align_up(anc_off + npad_max * max_depth * 4, 16);
        g_off = align_up(eg_off + npad_max * 4, 16);
        par_off = align_up(g_off + npad_max * 4, 16);
        dep_off = align_up(par_off + npad_max * 4, 16);
        poff_off = align_up(dep_off + npad_max * 4, 16);          // first pair of each node
        pnode_off = align_up(poff_off + (npad_max + 1) * 4, 16);  // node of each pair (u8)
        bar_off = align_up(pnode_off + npad_max * max_depth, 16);
        misc_off = bar_off + 8 * 8;
        pk_off = align_up(misc_off + 16, 16);
        if (pend_depth > 0) {
            pv_off = pk_off + pend_depth * dk * 4;
            pg_off = pv_off + pend_depth * dv * 4;
            ppath_off = pg_off + kMaxDepth * 4;
            pmisc_off = ppath_off + kMaxDepth * 4;
            total = align_up(pmisc_off + 32, 16) + 1024;
        } else {
            pv_off = pg_off = ppath_off = pmisc_off = pk_off;
            total = pk_off + 1024;  // + slack for 1024-byte base alignment
        }
    }
};

struct TcParams {
    VerifyArgs a;
    int npad_max;
    int tmem_cols;
    PendingArgs pend;  // commit + verify only
    float *H_w;        // the state rows written back (commit + verify only)
};

template <int DV, bool DIAG>
__global__ void __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_g, const TcParams P) {
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int dk = a.dk, H = a.H, md = a.max_depth;
    const TcLayout L(dk, DV, P.npad_max, md, DIAG);
    const uint32_t slab_bytes = P.npad_max * 128;
    uint8_t *sA = smem + L.a_off;
    uint8_t *sB = smem + L.b_off;
    uint8_t *sBlo = smem + L.blo_off;
    const __nv_bfloat16 *sQ = reinterpret_cast<const __nv_bfloat16 *>(smem + L.q_off);
    const __nv_bfloat16 *sK = reinterpret_cast<const __nv_bfloat16 *>(smem + L.k_off);
    const __nv_bfloat16 *sV = reinterpret_cast<const __nv_bfloat16 *>(smem + L.v_off);
    float *sE = reinterpret_cast<float *>(smem + L.e_off);
    float *sX = reinterpret_cast<float *>(smem + L.x_off);
    float *sW = reinterpret_cast<float *>(smem + L.w_off);
    int *sAnc = reinterpret_cast<int *>(smem + L.anc_off);
    float *sEG = reinterpret_cast<float *>(smem + L.eg_off);
    float *sG = reinterpret_cast<float *>(smem + L.g_off);
    int *sPar = reinterpret_cast<int *>(smem + L.par_off);
    int *sDep = reinterpret_cast<int *>(smem + L.dep_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sFlag = reinterpret_cast<int *>(smem + L.misc_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, b = unit / H, h = unit % H;
    const int nchunks = dk / kChunkRows;
    const uint32_t chunk_bytes = kChunkRows * DV * 4;  // fp32 in == bf16 hi + lo out
    // barriers: 0..3 H0 chunks, 4 factor tiles, 5 MMA completion
    const uint32_t bar0 = ptx::smem_addr(&bars[0]);
    const uint32_t bar_in = ptx::smem_addr(&bars[kMaxChunks]);
    const uint32_t bar_mma = ptx::smem_addr(&bars[kMaxChunks + 1]);

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        if (DIAG) ptx::prefetch_tensormap(&tm_g);
        for (int c = 0; c < kMaxChunks + 2; ++c) ptx::mbar_init(bar0 + 8 * c, 1);
        ptx::fence_mbar_init();
        *sFlag = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), P.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *sTmem;

    // inputs may be written by the previous kernel in the stream
    ptx::grid_dependency_wait();
    if (tid == 0) {
        // H0 (contiguous dk x DV fp32) streams in as row chunks, each on its own barrier
        const float *src = a.H0 + (size_t)unit * dk * DV;
        for (int c = 0; c < nchunks; ++c) {
            ptx::mbar_arrive_expect_tx(bar0 + 8 * c, chunk_bytes);
            ptx::bulk_g2s(ptx::smem_addr(sA) + c * chunk_bytes, src + c * kChunkRows * DV,
                          chunk_bytes, bar0 + 8 * c);
        }
    }

    int off = 0, n = 0;
    const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    if (!range_ok && tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
    const int npad = (n + 15) & ~15;
    const int slabs = dk / 64;
    const bool have_nodes = range_ok && n > 0;
    if (have_nodes && tid == 0) {
        const uint32_t rows_bf16 = npad * dk * 2;  // q or k bytes
        const uint32_t bytes = 2 * rows_bf16 + npad * DV * 2 + (DIAG ? npad * dk * 4 : 0);
        ptx::mbar_arrive_expect_tx(bar_in, bytes);
        for (int r = 0; r < npad; r += 16) {
            if (DIAG) {
                ptx::tma_load_3d(ptx::smem_addr(sQ) + r * dk * 2, &tm_q, 0, h, off + r, bar_in);
                ptx::tma_load_3d(ptx::smem_addr(sE) + r * dk * 4, &tm_g, 0, h, off + r, bar_in);
            } else {
                for (int s = 0; s < slabs; ++s)
                    ptx::tma_load_3d(ptx::smem_addr(sB + s * slab_bytes + r * 128), &tm_q, s * 64,
                                     h, off + r, bar_in);
            }
            ptx::tma_load_3d(ptx::smem_addr(sK) + r * dk * 2, &tm_k, 0, h, off + r, bar_in);
            ptx::tma_load_3d(ptx::smem_addr(sV) + r * DV * 2, &tm_v, 0, h, off + r, bar_in);
        }
    }
    ptx::grid_launch_dependents();

    // ---- this thread's tree entry (n <= 256 = blockDim), loaded while H0 lands
    int t_par = 0, t_dep = 0;
    float t_g = 0.f;
    if (have_nodes && tid < n) {
        t_par = a.parent[off + tid];
        t_dep = a.depth[off + tid];
        if (!DIAG) t_g = a.g[(size_t)(off + tid) * H + h];
    }

    // ---- H0: once every chunk has landed, split it in place into bf16 hi/lo K-major
    // operand rows.  Chunk layout (kChunkRows keys): operand rows (value channels) in
    // 8-row groups of 512 bytes (4 core matrices of 8 rows x 8 keys); DV = 64 stacks
    // hi rows 0..63 over lo rows 64..127; DV = 128 keeps a hi and a lo operand of 128
    // rows, 8 KB each.
    constexpr int kPerChunk = DV * (kChunkRows / 8) / kThreads;  // items per thread per chunk
    float hold[kMaxChunks][kPerChunk][8];
    // one thread waits on the copies; the others park at the block barrier
    bool got = true;
    if (tid == 0) {
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c)
            if (c < nchunks) got = ptx::mbar_wait(bar0 + 8 * c, 0, kWaitLimit) && got;
    }
    if (have_nodes && tid < n) {  // tree entry to shared memory; parents must precede
        sPar[tid] = t_par;
        sDep[tid] = t_dep;
        if (!DIAG) sG[tid] = t_g;
        if (t_par < -1 || t_par >= tid) *sFlag = 1;
    }
    got = __syncthreads_and(got);
    if (got) {
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            if (c >= nchunks) break;
            const float *f32 = reinterpret_cast<const float *>(sA + c * chunk_bytes);
#pragma unroll
            for (int t = 0; t < kPerChunk; ++t) {
                const int it = tid + t * kThreads;
                const int ch = it % DV, kq = it / DV;
#pragma unroll
                for (int e = 0; e < 8; ++e) hold[c][t][e] = f32[(kq * 8 + e) * DV + ch];
            }
        }
    }
    __syncthreads();  // every H0 read is done before the in-place rewrite
    bool run = got;
    if (!run && tid == 0) report(a.status, TV_ERR_TIMEOUT);
    run = run && have_nodes;
    if (run) {
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            if (c >= nchunks) break;
            uint8_t *chunk = sA + c * chunk_bytes;
#pragma unroll
            for (int t = 0; t < kPerChunk; ++t) {
                const int it = tid + t * kThreads;
                const int ch = it % DV, kq = it / DV;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split_pair(hold[c][t][2 * e], hold[c][t][2 * e + 1], hi[e], lo[e]);
                const int r_hi = ch;
                const int r_lo = DV == 64 ? 64 + ch : ch;
                uint8_t *lo_base = DV == 64 ? chunk : chunk + 8192;
                *reinterpret_cast<uint4 *>(chunk + (r_hi / 8) * 512 + kq * 128 + (r_hi % 8) * 16) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(lo_base + (r_lo / 8) * 512 + kq * 128 + (r_lo % 8) * 16) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();

    // D[c][i] = sum_r A[c][r] B[i][r] on the tensor core, one thread issues
    auto issue_mma = [&]() {
        const uint32_t idesc = ptx::idesc_bf16_f32(128, npad);
        const uint32_t b_hi = ptx::smem_addr(sB), b_lo = ptx::smem_addr(sBlo);
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t a_hi = ptx::smem_addr(sA + c * chunk_bytes);
            const uint32_t a_lo = DV == 64 ? a_hi : a_hi + 8192;
            uint32_t pa[3], pb[3];
            int npass = 0;
            pa[npass] = a_hi; pb[npass++] = b_hi;  // DV = 64: hi and lo rows together
            if (DV == 128) { pa[npass] = a_lo; pb[npass++] = b_hi; }
            if (DIAG) { pa[npass] = a_hi; pb[npass++] = b_lo; }
            for (int p = 0; p < npass; ++p) {
                for (int s2 = 0; s2 < kChunkRows / 16; ++s2) {
                    const int kk = c * (kChunkRows / 16) + s2;  // global 16-key step
                    const uint64_t ad = ptx::desc_kmajor_noswizzle(pa[p] + s2 * 256, 128, 512);
                    const uint64_t bd = ptx::desc_kmajor_sw128(
                        pb[p] + (kk / 4) * slab_bytes + (kk % 4) * 32, 1024);
                    ptx::mma_bf16(tmem, ad, bd, idesc, (c > 0 || p > 0 || s2 > 0) ? 1u : 0u);
                }
            }
        }
        ptx::mma_commit(bar_mma);
    };

    // ---- factor tiles: the scalar-decay context term needs only q, so its MMAs go
    // out now and run under the tree checks and ancestor scores
    bool landed = true;
    if (tid == 0 && have_nodes) landed = ptx::mbar_wait(bar_in, 0, kWaitLimit);
    if (!DIAG && run && tid == 0 && landed) issue_mma();
    // tree: depth[i] = depth[parent] + 1 (1 at the context), within max_depth
    if (have_nodes && tid < n && *sFlag == 0) {
        const int want = t_par < 0 ? 1 : sDep[t_par] + 1;
        if (t_dep != want || t_dep > md) *sFlag = 1;
    }
    const bool all_landed = __syncthreads_and(landed);
    bool mma_issued = !DIAG && run && all_landed;
    if (!all_landed && tid == 0 && run) report(a.status, TV_ERR_TIMEOUT);
    const bool tree_ok = *sFlag == 0;
    if (have_nodes && !tree_ok) {
        for (int e = tid; e < n * DV; e += kThreads)
            a.out[((size_t)(off + e / DV) * H + h) * DV + e % DV] = 0.f;
        if (tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
    }
    run = run && all_landed && tree_ok;

    if (DIAG && run) {
        for (int e = tid; e < n * dk; e += kThreads) sE[e] = expf(sE[e]);
        __syncthreads();
    }
    if (run && !DIAG) {
        // root path of each node with the decay factor of every (node, ancestor) pair:
        // anc_d(i) = the ancestor d steps up, e^{G_i - G_{anc_d}} = exp(sum of g over the
        // path nodes below it), and e^{G_i}
        if (tid < n) {
            float s = 0.f;
            int j = tid, d = 0;
            while (j >= 0) {
                sAnc[tid * md + d] = j;
                sW[tid * md + d] = expf(s);
                s += sG[j];
                j = sPar[j];
                ++d;
            }
            sEG[tid] = expf(s);
        }
        __syncthreads();
        // w_ij = decay * (q_i . k_j): one 8-lane group per node, its ancestors in turn.
        // Loop bounds are uniform across the warp (the shuffles need every lane).
        const int sub = lane & 7;
        const int per = dk / 8;  // 16 or 8 key channels per lane, whole 16-byte chunks
        for (int base = warp * 4; base < n; base += kThreads / 8) {
            const int i = base + (lane >> 3);
            const bool valid = i < n;
            float qv[16];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (valid && u * 8 < per) {
                    const int c = sub * per + u * 8;
                    const uint4 raw = *reinterpret_cast<const uint4 *>(sB + swz_offset(i, c, slab_bytes));
                    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        qv[u * 8 + 2 * e] = __low2float(p2[e]);
                        qv[u * 8 + 2 * e + 1] = __high2float(p2[e]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) qv[u * 8 + e] = 0.f;
                }
            }
            const int di = valid ? sDep[i] : 0;
            const int dmax = __reduce_max_sync(0xffffffffu, di);
            for (int d = 0; d < dmax; ++d) {
                const bool act = d < di;
                float part = 0.f;
                if (act) {
                    const int j = sAnc[i * md + d];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (u * 8 < per) {
                            const uint4 raw = *reinterpret_cast<const uint4 *>(sK + j * dk + sub * per + u * 8);
                            const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                part += qv[u * 8 + 2 * e] * __low2float(p2[e]) +
                                        qv[u * 8 + 2 * e + 1] * __high2float(p2[e]);
                        }
                    }
                }
                part += __shfl_xor_sync(0xffffffffu, part, 4);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                if (act && sub == 0) sW[i * md + d] *= part;
            }
        }
    }
    if (run && DIAG) {
        // one warp per node walks its root path with a per-channel decay product
        const int per_lane = dk / 32;    // 2 or 4 key channels per lane
        const int c0 = lane * per_lane;  // within one 16-byte chunk
        for (int i = warp; i < n; i += kThreads / 32) {
            float qv[4];
            load_bf16x(sQ + i * dk + c0, per_lane, qv);
            float f[4] = {1.f, 1.f, 1.f, 1.f};  // e^{G_i - G_j} per channel
            int j = i, d = 0;
            while (j >= 0) {
                float kv[4];
                load_bf16x(sK + j * dk + c0, per_lane, kv);
                float part = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) part += qv[m] * kv[m] * f[m];
                part = warp_sum(part);
                if (lane == 0) {
                    sW[i * md + d] = part;
                    sAnc[i * md + d] = j;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (m < per_lane) f[m] *= sE[j * dk + c0 + m];
                j = sPar[j];
                ++d;
            }
            // B = bf16 hi/lo of e^{G_i} * q_i in the swizzled K-major layout
            uint32_t hi[2], lo[2];
            split_pair(qv[0] * f[0], qv[1] * f[1], hi[0], lo[0]);
            split_pair(qv[2] * f[2], qv[3] * f[3], hi[1], lo[1]);
            const uint32_t o = swz_offset(i, c0, slab_bytes);
            if (per_lane == 4) {
                *reinterpret_cast<uint2 *>(sB + o) = make_uint2(hi[0], hi[1]);
                *reinterpret_cast<uint2 *>(sBlo + o) = make_uint2(lo[0], lo[1]);
            } else {
                *reinterpret_cast<uint32_t *>(sB + o) = hi[0];
                *reinterpret_cast<uint32_t *>(sBlo + o) = lo[0];
            }
        }
        // rows n..npad-1 of B feed unused output columns; keep them finite
        for (int e = n * 64 + tid; e < npad * 64; e += kThreads) {
            const int i = e / 64, cq = (e % 64) * 2;
            const uint32_t o = swz_offset(i, cq, slab_bytes);
            if (cq < dk) {
                *reinterpret_cast<uint32_t *>(sB + o) = 0u;
                *reinterpret_cast<uint32_t *>(sBlo + o) = 0u;
            }
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (DIAG && run && tid == 0) issue_mma();
    if (DIAG) mma_issued = run;

    // ---- wait for the tensor core (always, once its MMAs are out)
    bool mma_ok = true;
    if (mma_issued && tid == 0) mma_ok = ptx::mbar_wait(bar_mma, 0, kWaitLimit);
    const bool all_mma = __syncthreads_and(mma_ok);
    if (mma_issued && !all_mma && tid == 0) report(a.status, TV_ERR_TIMEOUT);
    run = run && all_mma;
    ptx::tc_fence_after_sync();

    // after a timed-out wait, give the copies one more bounded wait before the CTA
    // (and its shared memory) goes away
    if (tid == 0 && !got)
        for (int c = 0; c < nchunks; ++c) ptx::mbar_wait(bar0 + 8 * c, 0, kWaitLimit);
    if (tid == 0 && have_nodes && !all_landed) ptx::mbar_wait(bar_in, 0, kWaitLimit);

    // ---- epilogue: o_i = [e^{G_i}] * D[:, i] + sum_d w_{i,d} v_{anc_d(i)}
    auto ancestor_sum = [&](int i, int c, float o) {
        const int di = sDep[i];
        const int *ap = sAnc + i * md;
        const float *wp = sW + i * md;
        for (int d0 = 0; d0 < di; d0 += 4) {
            int jj[4];
            float ww[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool in = d0 + u < di;
                jj[u] = in ? ap[d0 + u] : 0;
                ww[u] = in ? wp[d0 + u] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) o += ww[u] * __bfloat162float(sV[jj[u] * DV + c]);
        }
        return o;
    };
    const int quad = warp & 3, half = warp >> 2;
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    if (DV == 64) {
        // every warp dumps its quadrant (hi rows 0..63, lo rows 64..127) for half the
        // columns; then all threads form outputs (node, channel), channels fastest
        const int ncols_half = npad / 2;  // multiple of 8
        if (run) {
            const int row = 32 * quad + lane;
            for (int col = half * ncols_half; col < (half + 1) * ncols_half; col += 8) {
                float vals[8];
                ptx::tmem_ld_x8(tq + col, vals);
#pragma unroll
                for (int e = 0; e < 8; ++e) sX[(col + e) * 128 + row] = vals[e];
            }
        }
        __syncthreads();
        if (run) {
            const int c = tid & 63;
            for (int i = tid >> 6; i < n; i += kThreads / 64) {
                float o = sX[i * 128 + c] + sX[i * 128 + 64 + c];
                if (!DIAG) o *= sEG[i];
                a.out[((size_t)(off + i) * H + h) * DV + c] = ancestor_sum(i, c, o);
            }
        }
    } else if (run) {
        const int ncols_half = npad / 2;
        const int c = 32 * quad + lane;
        for (int col = half * ncols_half; col < (half + 1) * ncols_half; col += 8) {
            float vals[8];
            ptx::tmem_ld_x8(tq + col, vals);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = col + e;
                if (i >= n) break;
                float o = vals[e];
                if (!DIAG) o *= sEG[i];
                a.out[((size_t)(off + i) * H + h) * DV + c] = ancestor_sum(i, c, o);
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// Scalar-decay verification, warp-specialized so that independent phases overlap:
//   warps 0-3 stream H0 in chunks, split each chunk in place into bf16 hi/lo operand
//     rows as it lands, then issue the context MMA (D = H0^T q) as soon as q has landed;
//   warps 4-7 read the request's offsets and tree, issue the q/k/v tile copies,
//     validate the tree and compute the ancestor scores
//     w_{i,d} = e^{G_i - G_{anc_d(i)}} (q_i . k_{anc_d(i)}) and e^{G_i};
//   all eight warps then form o_i = e^{G_i} D[:, i] + sum_d w_{i,d} v_{anc_d(i)}.
// Same shared-memory plan, operand layouts and error behaviour as verify_tc_kernel.
//
// PEND (tv_commit_verify): before the state is split, the previous step's accepted
// path p_1..p_L is applied to it (Bole summary page, "Core techniques" §2):
//   H[r][c] <- e^{G_L} H[r][c] + sum_m e^{G_L - G_{p_m}} k_{p_m}[r] v_{p_m}[c],
// the updated rows are written back to the state in HBM and the context term is
// formed from them.  The H0 group reads the path and gathers its factor rows while
// the first chunk is in flight; a request with L = 0 writes nothing.
// Residency at dv = 64: 45 KB of shared memory per CTA at 16-node trees, so four
// CTAs fit an SM and registers are capped to match (the launch asks for the whole
// shared-memory carveout); the pending-commit variant keeps three.
template <int DV, bool PEND>
__global__ void __launch_bounds__(kThreads, PEND ? 3 : (DV == 64 ? 4 : 1))
    verify_tc_scalar_ws_kernel(const __grid_constant__ CUtensorMap tm_q,
                               const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v, const TcParams P) {
    constexpr int kGroup = kThreads / 2;  // threads per specialized group
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int dk = a.dk, H = a.H, md = a.max_depth;
    const TcLayout L(dk, DV, P.npad_max, md, false, PEND ? P.pend.max_depth : 0);
    const uint32_t slab_bytes = P.npad_max * 128;
    uint8_t *sA = smem + L.a_off;
    uint8_t *sB = smem + L.b_off;
    const __nv_bfloat16 *sK = reinterpret_cast<const __nv_bfloat16 *>(smem + L.k_off);
    const __nv_bfloat16 *sV = reinterpret_cast<const __nv_bfloat16 *>(smem + L.v_off);
    float *sX = reinterpret_cast<float *>(smem + L.x_off);
    // per (node, ancestor) pair p, numbered node by node (sPairOff): the ancestor,
    // its weight w_p and its node
    float *sW = reinterpret_cast<float *>(smem + L.w_off);
    int *sAnc = reinterpret_cast<int *>(smem + L.anc_off);
    float *sEG = reinterpret_cast<float *>(smem + L.eg_off);
    float *sG = reinterpret_cast<float *>(smem + L.g_off);
    int *sPar = reinterpret_cast<int *>(smem + L.par_off);
    int *sDep = reinterpret_cast<int *>(smem + L.dep_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sFlag = reinterpret_cast<int *>(smem + L.misc_off + 4);   // tree error
    int *sState = reinterpret_cast<int *>(smem + L.misc_off + 8);  // copy/MMA progress bits
    int *sPairOff = reinterpret_cast<int *>(smem + L.poff_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, b = unit / H, h = unit % H;
    const int nchunks = dk / kChunkRows;
    const uint32_t chunk_bytes = kChunkRows * DV * 4;
    const uint32_t bar0 = ptx::smem_addr(&bars[0]);
    const uint32_t bar_in = ptx::smem_addr(&bars[kMaxChunks]);
    const uint32_t bar_mma = ptx::smem_addr(&bars[kMaxChunks + 1]);
    // progress bits; each is written by one group only, before that group's barrier
    enum { kH0Late = 1, kQkvLateTree = 2, kMmaOut = 4, kQkvLateMma = 8 };

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        for (int c = 0; c < kMaxChunks + 2; ++c) ptx::mbar_init(bar0 + 8 * c, 1);
        ptx::fence_mbar_init();
        *sFlag = 0;
        *sState = 0;
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
    if (tid == 0) {
        const float *src = a.H0 + (size_t)unit * dk * DV;
        for (int c = 0; c < nchunks; ++c) {
            ptx::mbar_arrive_expect_tx(bar0 + 8 * c, chunk_bytes);
            ptx::bulk_g2s(ptx::smem_addr(sA) + c * chunk_bytes, src + c * kChunkRows * DV,
                          chunk_bytes, bar0 + 8 * c);
        }
    }
    int off = 0, n = 0;
    const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    const int npad = (n + 15) & ~15;
    const bool have_nodes = range_ok && n > 0;
    ptx::grid_launch_dependents();

    if (warp < 4) {
        // ================= H0 group: split chunks as they land, then the MMA
        constexpr int kPer = DV * (kChunkRows / 8) / kGroup;  // (channel, 8-key) items
        // pending commit: path length pL, e^{G_L} and the path's scaled factor rows
        int pL = 0;
        float palpha = 1.f;
        float *sPK = reinterpret_cast<float *>(smem + L.pk_off);  // [pL][dk] e^{G_L-G_m} k_m
        float *sPV = reinterpret_cast<float *>(smem + L.pv_off);  // [pL][DV] v_m
        if constexpr (PEND) {
            const PendingArgs &pa = P.pend;
            const int mdp = pa.max_depth;
            float *sPG = reinterpret_cast<float *>(smem + L.pg_off);
            int *sPath = reinterpret_cast<int *>(smem + L.ppath_off);
            // L, bad range/length/entry, offset, not a root path, e^{G_L} (float bits)
            int *sPM = reinterpret_cast<int *>(smem + L.pmisc_off);
            if (warp == 0) {
                int poff = 0, pn = 0;
                const bool prange =
                    request_range(pa.node_offsets, b, pa.T, pa.max_nodes, poff, pn);
                const int Lp = pa.len[b];
                const int pnode = lane < mdp ? pa.path[(size_t)b * mdp + lane] : -1;
                bool bad = !prange || Lp < 0 || Lp > mdp || (lane < Lp && (pnode < 0 || pnode >= pn));
                bad = __any_sync(0xffffffffu, bad);
                if (!bad && lane < Lp) sPath[lane] = pnode;
                if (lane == 0) {
                    sPM[0] = bad ? 0 : Lp;
                    sPM[1] = bad;
                    sPM[2] = poff;
                    sPM[3] = 0;
                }
            }
            named_barrier(1, kGroup);
            const int Lp = sPM[0], poff = sPM[2];
            if (Lp > 0) {
                // the path must be a root path of the previous tree; its factor rows
                if (warp == 0) {
                    bool bad = false;
                    if (lane < Lp)
                        bad = pa.parent[poff + sPath[lane]] != (lane == 0 ? -1 : sPath[lane - 1]);
                    bad = __any_sync(0xffffffffu, bad);
                    if (lane == 0) sPM[3] = bad;
                }
                const __nv_bfloat16 *pk = static_cast<const __nv_bfloat16 *>(pa.k);
                const __nv_bfloat16 *pv = static_cast<const __nv_bfloat16 *>(pa.v);
                const int k8 = dk / 8, v8 = DV / 8;
                for (int e = tid; e < Lp * (k8 + v8); e += kGroup) {
                    const bool isk = e < Lp * k8;
                    const int e2 = isk ? e : e - Lp * k8;
                    const int per = isk ? k8 : v8;
                    const int m = e2 / per, c8 = (e2 % per) * 8;
                    const size_t row = (size_t)(poff + sPath[m]) * H + h;
                    const uint4 raw = *reinterpret_cast<const uint4 *>(
                        isk ? pk + row * dk + c8 : pv + row * DV + c8);
                    const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                    float *dst = isk ? sPK + m * dk + c8 : sPV + m * DV + c8;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        dst[2 * u] = __low2float(x2[u]);
                        dst[2 * u + 1] = __high2float(x2[u]);
                    }
                }
                if (tid < Lp) sPG[tid] = pa.g[(size_t)(poff + sPath[tid]) * H + h];
                named_barrier(1, kGroup);
                if (sPM[3] == 0) {
                    // a_{m,r} = e^{sum of g after p_m} k_{p_m}[r]; e^{G_L} once per row
                    for (int r = tid; r < dk; r += kGroup) {
                        float sg = 0.f;
                        for (int m = Lp - 1; m >= 0; --m) {
                            sPK[m * dk + r] *= expf(sg);
                            sg += sPG[m];
                        }
                        if (r == 0) reinterpret_cast<float *>(sPM)[4] = expf(sg);
                    }
                }
                named_barrier(1, kGroup);
                if (sPM[3] == 0) {
                    pL = Lp;
                    palpha = reinterpret_cast<const float *>(sPM)[4];
                }
            }
        }
        float *Hw = PEND ? P.H_w + (size_t)unit * dk * DV : nullptr;
        // the pending update makes the loop body long: keep one copy of it in the
        // instruction cache
        constexpr int kUnrollChunks = PEND ? 1 : kMaxChunks;
#pragma unroll kUnrollChunks
        for (int c = 0; c < kMaxChunks; ++c) {
            if (c >= nchunks) break;
            if (tid == 0 && !ptx::mbar_wait(bar0 + 8 * c, 0, kWaitLimit)) atomicOr(sState, kH0Late);
            named_barrier(1, kGroup);
            const bool landed = (*sState & kH0Late) == 0;
            const bool ok = landed && have_nodes;
            uint8_t *chunk = sA + c * chunk_bytes;
            float hold[kPer][8];
            if (landed && (have_nodes || pL > 0)) {
                const float *f32 = reinterpret_cast<const float *>(chunk);
#pragma unroll
                for (int t = 0; t < kPer; ++t) {
                    const int it = tid + t * kGroup;
                    const int ch = it % DV, kq = it / DV;
#pragma unroll
                    for (int e = 0; e < 8; ++e) hold[t][e] = f32[(kq * 8 + e) * DV + ch];
                }
            }
            if (PEND && landed && pL > 0) {
                // the pending rank-pL update; each thread owns 8 consecutive rows x 1
                // channel per item, so a warp's stores of one row are 128 contiguous bytes
#pragma unroll
                for (int t = 0; t < kPer; ++t)
#pragma unroll
                    for (int e = 0; e < 8; ++e) hold[t][e] *= palpha;
                for (int m = 0; m < pL; ++m) {
#pragma unroll
                    for (int t = 0; t < kPer; ++t) {
                        const int it = tid + t * kGroup;
                        const int ch = it % DV, kq = it / DV;
                        const float vm = sPV[m * DV + ch];
                        const float4 k0 = *reinterpret_cast<const float4 *>(
                            sPK + m * dk + c * kChunkRows + kq * 8);
                        const float4 k1 = *reinterpret_cast<const float4 *>(
                            sPK + m * dk + c * kChunkRows + kq * 8 + 4);
                        hold[t][0] += k0.x * vm; hold[t][1] += k0.y * vm;
                        hold[t][2] += k0.z * vm; hold[t][3] += k0.w * vm;
                        hold[t][4] += k1.x * vm; hold[t][5] += k1.y * vm;
                        hold[t][6] += k1.z * vm; hold[t][7] += k1.w * vm;
                    }
                }
#pragma unroll
                for (int t = 0; t < kPer; ++t) {
                    const int it = tid + t * kGroup;
                    const int ch = it % DV, kq = it / DV;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        Hw[(size_t)(c * kChunkRows + kq * 8 + e) * DV + ch] = hold[t][e];
                }
            }
            named_barrier(1, kGroup);  // the chunk is read before it is rewritten in place
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
                    *reinterpret_cast<uint4 *>(lo_base + (r_lo / 8) * 512 + kq * 128 + (r_lo % 8) * 16) =
                        make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        named_barrier(1, kGroup);
        ptx::tc_fence_after_sync();
        if (tid == 0 && have_nodes && (*sState & kH0Late) == 0) {
            if (ptx::mbar_wait(bar_in, 0, kWaitLimit)) {
                const uint32_t idesc = ptx::idesc_bf16_f32(128, npad);
                const uint32_t b0 = ptx::smem_addr(sB);
                for (int c = 0; c < nchunks; ++c) {
                    const uint32_t a_hi = ptx::smem_addr(sA + c * chunk_bytes);
                    const int npass = DV == 64 ? 1 : 2;  // DV = 128: hi operand, then lo
                    for (int p = 0; p < npass; ++p) {
                        const uint32_t a_op = a_hi + p * 8192;
                        for (int s2 = 0; s2 < kChunkRows / 16; ++s2) {
                            const int kk = c * (kChunkRows / 16) + s2;
                            const uint64_t ad = ptx::desc_kmajor_noswizzle(a_op + s2 * 256, 128, 512);
                            const uint64_t bd = ptx::desc_kmajor_sw128(
                                b0 + (kk / 4) * slab_bytes + (kk % 4) * 32, 1024);
                            ptx::mma_bf16(tmem, ad, bd, idesc, (c > 0 || p > 0 || s2 > 0) ? 1u : 0u);
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
        // ================= tree group: tree, factor tiles, ancestor scores
        const int t = tid - kGroup;
        if (t == 0 && have_nodes) {
            const int slabs = dk / 64;
            ptx::mbar_arrive_expect_tx(bar_in, 2 * npad * dk * 2 + npad * DV * 2);
            for (int r = 0; r < npad; r += 16) {
                for (int s = 0; s < slabs; ++s)
                    ptx::tma_load_3d(ptx::smem_addr(sB + s * slab_bytes + r * 128), &tm_q, s * 64,
                                     h, off + r, bar_in);
                ptx::tma_load_3d(ptx::smem_addr(sK) + r * dk * 2, &tm_k, 0, h, off + r, bar_in);
                ptx::tma_load_3d(ptx::smem_addr(sV) + r * DV * 2, &tm_v, 0, h, off + r, bar_in);
            }
        }
        if (have_nodes) {
            for (int i = t; i < n; i += kGroup) {
                const int p = a.parent[off + i], d = a.depth[off + i];
                const float gv = a.g[(size_t)(off + i) * H + h];
                sPar[i] = p;
                sDep[i] = d;
                sG[i] = gv;
                if (p < -1 || p >= i) *sFlag = 1;
            }
        }
        named_barrier(2, kGroup);
        if (have_nodes && *sFlag == 0)
            for (int i = t; i < n; i += kGroup) {
                const int p = sPar[i];
                const int want = p < 0 ? 1 : sDep[p] + 1;
                if (sDep[i] != want || sDep[i] > md) *sFlag = 1;
            }
        named_barrier(2, kGroup);
        const bool tree_ok = have_nodes && *sFlag == 0;
        if (tree_ok && warp == 4) {
            // (node, ancestor) pairs numbered node by node: exclusive scan of depths
            const int per = (n + 31) / 32;
            int local = 0;
            for (int u = 0; u < per; ++u) {
                const int i = lane * per + u;
                if (i < n) local += sDep[i];
            }
            int incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int run_sum = incl - local;
            for (int u = 0; u < per; ++u) {
                const int i = lane * per + u;
                if (i < n) {
                    sPairOff[i] = run_sum;
                    run_sum += sDep[i];
                }
            }
            if (lane == 31) sPairOff[n] = incl;
        }
        named_barrier(2, kGroup);
        uint8_t *sPairNode = smem + L.pnode_off;
        if (tree_ok) {
            // root paths with the decay factor of every (node, ancestor) pair:
            // anc_d(i), e^{G_i - G_{anc_d(i)}} and e^{G_i}; needs only the tree and g
            for (int i = t; i < n; i += kGroup) {
                float s = 0.f;
                int j = i, d = 0;
                const int p0 = sPairOff[i];
                while (j >= 0) {
                    sAnc[p0 + d] = j;
                    sW[p0 + d] = expf(s);
                    sPairNode[p0 + d] = static_cast<uint8_t>(i);
                    s += sG[j];
                    j = sPar[j];
                    ++d;
                }
                sEG[i] = expf(s);
            }
        }
        if (t == 0 && have_nodes && !ptx::mbar_wait(bar_in, 0, kWaitLimit))
            atomicOr(sState, kQkvLateTree);
        named_barrier(2, kGroup);
        if (tree_ok && (*sState & kQkvLateTree) == 0) {
            pair_scores(sB, sK, sPairOff, sPairNode, sAnc, sW, n, dk, slab_bytes,
                        (warp - 4) * 4 + (lane >> 3), lane);
        }
    }

    // ================= join
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const int st = *sState;
    const bool tree_ok = *sFlag == 0;
    const bool mma_out = (st & kMmaOut) != 0;
    if (tid == 0) {
        if (!range_ok && h == 0) report(a.status, TV_ERR_TREE);
        if (have_nodes && !tree_ok && h == 0) report(a.status, TV_ERR_TREE);
        if (st & (kH0Late | kQkvLateTree | kQkvLateMma)) report(a.status, TV_ERR_TIMEOUT);
        if constexpr (PEND) {
            const int *sPM = reinterpret_cast<const int *>(smem + L.pmisc_off);
            if ((sPM[1] || sPM[3]) && h == 0) report(a.status, TV_ERR_TREE);
        }
    }
    if (have_nodes && !tree_ok)
        for (int e = tid; e < n * DV; e += kThreads)
            a.out[((size_t)(off + e / DV) * H + h) * DV + e % DV] = 0.f;
    bool mma_ok = true;
    if (mma_out && tid == 0) mma_ok = ptx::mbar_wait(bar_mma, 0, kWaitLimit);
    mma_ok = __syncthreads_and(mma_ok);
    if (mma_out && !mma_ok && tid == 0) report(a.status, TV_ERR_TIMEOUT);
    ptx::tc_fence_after_sync();
    const bool run = have_nodes && tree_ok && mma_out && mma_ok && !(st & kQkvLateTree);

    // ---- epilogue, 32 node columns at a time: every warp copies its tensor-memory
    // quadrant (rows = value channels; dv = 64 keeps hi rows 0-63 and lo rows 64-127)
    // into shared memory; then each thread forms 4 consecutive channels of one node:
    // o_i = e^{G_i} D[:, i] + sum_d w_{i,d} v_{anc_d(i)}, stored as a float4
    float *sXc = reinterpret_cast<float *>(sA);  // A is free once the MMAs completed
    const int quad = warp & 3, half = warp >> 2;
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    constexpr int kQuads = DV / 4;
    for (int c0 = 0; c0 < npad; c0 += 32) {  // npad is uniform
        const int ncol = min(32, npad - c0);  // 16 or 32
        if (run) {
            const int row = 32 * quad + lane;
            for (int col = half * (ncol / 2); col < (half + 1) * (ncol / 2); col += 8) {
                float vals[8];
                ptx::tmem_ld_x8(tq + c0 + col, vals);
#pragma unroll
                for (int e = 0; e < 8; ++e) sXc[(col + e) * 128 + row] = vals[e];
            }
        }
        __syncthreads();
        if (run) {
            const int ntask = min(ncol, n - c0) * kQuads;
            for (int task = tid; task < ntask; task += kThreads) {
                const int il = task / kQuads, c = (task % kQuads) * 4;
                const int i = c0 + il;
                float4 o = *reinterpret_cast<const float4 *>(sXc + il * 128 + c);
                if (DV == 64) {
                    const float4 lo = *reinterpret_cast<const float4 *>(sXc + il * 128 + 64 + c);
                    o.x += lo.x; o.y += lo.y; o.z += lo.z; o.w += lo.w;
                }
                const float eg = sEG[i];
                o.x *= eg; o.y *= eg; o.z *= eg; o.w *= eg;
                const int di = sDep[i], p0 = sPairOff[i];
                for (int d = 0; d < di; ++d) {
                    const float w = sW[p0 + d];
                    const uint2 raw = *reinterpret_cast<const uint2 *>(sV + sAnc[p0 + d] * DV + c);
                    const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
                    const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
                    o.x += w * __low2float(v01); o.y += w * __high2float(v01);
                    o.z += w * __low2float(v23); o.w += w * __high2float(v23);
                }
                *reinterpret_cast<float4 *>(a.out + ((size_t)(off + i) * H + h) * DV + c) = o;
            }
        }
        __syncthreads();  // the staging buffer is reused by the next column chunk
    }

    // a timed-out copy gets one more bounded wait before the CTA's memory goes away
    if (tid == 0 && (st & kH0Late))
        for (int c = 0; c < nchunks; ++c) ptx::mbar_wait(bar0 + 8 * c, 0, kWaitLimit);
    if (tid == 0 && (st & (kQkvLateTree | kQkvLateMma))) ptx::mbar_wait(bar_in, 0, kWaitLimit);
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// ---------------------------------------------------------------- host side

size_t tc_smem_bytes(const VerifyArgs &a, int pend_depth = 0) {
    const int npad_max = (a.max_nodes + 15) & ~15;
    return TcLayout(a.dk, a.dv, npad_max, a.max_depth, a.decay == TV_DECAY_DIAG, pend_depth).total;
}

// Shared-memory opt-in, a residency cap that keeps co-resident CTAs within the 512
// tensor-memory columns of an SM, and a programmatic-dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_tc_kernel(void (*kern)(KArgs...), const TcParams &P, size_t smem,
                             unsigned grid, cudaStream_t s, Args &&...args) {
    cudaError_t e = configure_smem_once(kern, true);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    const int max_ctas = 512 / P.tmem_cols;
    if (per_sm > max_ctas) {
        // enlarge the request so that max_ctas + 1 blocks no longer fit on one SM
        int dev = 0, smem_sm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        const size_t need = (size_t)smem_sm / (max_ctas + 1) + 1;
        if (need > smem) smem = need;
    }
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, static_cast<Args &&>(args)...);
}

// PEND: the scalar kernel with the pending commit of *pend applied to H first.
template <int DV, bool DIAG, bool PEND = false>
cudaError_t launch_tc(const VerifyArgs &a, cudaStream_t s, const PendingArgs *pend = nullptr,
                      float *H = nullptr) {
    static_assert(!(DIAG && PEND), "the pending commit runs in the scalar-decay kernel");
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv_, tg;
    bool enc = encode_rows(&tk, a.k, BF, 2, a.dk, a.H, a.T, a.dk, CU_TENSOR_MAP_SWIZZLE_NONE) &&
               encode_rows(&tv_, a.v, BF, 2, DV, a.H, a.T, DV, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (DIAG) {
        enc = enc && encode_rows(&tq, a.q, BF, 2, a.dk, a.H, a.T, a.dk, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              encode_rows(&tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dk, a.H, a.T, a.dk,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        enc = enc && encode_rows(&tq, a.q, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        tg = tk;  // unused
    }
    if (!enc) return cudaErrorInvalidValue;

    TcParams P;
    P.a = a;
    P.npad_max = (a.max_nodes + 15) & ~15;
    P.tmem_cols = tmem_columns(P.npad_max);
    P.pend = pend ? *pend : PendingArgs{};
    P.H_w = H;
    const size_t smem = tc_smem_bytes(a, pend ? pend->max_depth : 0);
    const unsigned grid = (unsigned)(a.B * a.H);
    if constexpr (DIAG)
        return launch_tc_kernel(verify_tc_kernel<DV, true>, P, smem, grid, s, tq, tk, tv_, tg, P);
    else
        return launch_tc_kernel(verify_tc_scalar_ws_kernel<DV, PEND>, P, smem, grid, s, tq, tk,
                                tv_, P);
}

}  // namespace

bool verify_tc_supported(const VerifyArgs &a) {
    return a.qkv_dtype == TV_BF16 && (a.dk == 64 || a.dk == 128) && (a.dv == 64 || a.dv == 128) &&
           a.max_nodes <= kMaxNodes && tc_smem_bytes(a) <= kSmemLimit && encode_fn() != nullptr;
}

cudaError_t launch_verify_tc(const VerifyArgs &a, cudaStream_t s) {
    if (!verify_tc_supported(a)) return cudaErrorNotSupported;
    const bool diag = a.decay == TV_DECAY_DIAG;
    if (a.dv == 64) return diag ? launch_tc<64, true>(a, s) : launch_tc<64, false>(a, s);
    return diag ? launch_tc<128, true>(a, s) : launch_tc<128, false>(a, s);
}

bool commit_verify_tc_supported(const VerifyArgs &a, const PendingArgs &p) {
    return a.decay == TV_DECAY_SCALAR && verify_tc_supported(a) &&
           tc_smem_bytes(a, p.max_depth) <= kSmemLimit;
}

cudaError_t launch_commit_verify_tc(const VerifyArgs &a, const PendingArgs &p, float *H,
                                    cudaStream_t s) {
    if (!commit_verify_tc_supported(a, p)) return cudaErrorNotSupported;
    if (a.dv == 64) return launch_tc<64, false, true>(a, s, &p, H);
    return launch_tc<128, false, true>(a, s, &p, H);
}

}  // namespace tv
