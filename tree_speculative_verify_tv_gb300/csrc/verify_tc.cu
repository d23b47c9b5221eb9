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
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_ptx.cuh"
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kThreads = 256;
constexpr long long kWaitLimit = 2000000000LL;  // ~1 s at 2 GHz

__host__ __device__ constexpr uint32_t align_up(uint32_t x, uint32_t a) {
    return (x + a - 1) / a * a;
}

// Shared-memory plan, identical on host and device.  TMA destinations are
// 1024-byte aligned.
struct TcLayout {
    uint32_t a_off, q_off, k_off, v_off, x_off, w_off, eg_off, g_off, par_off, dep_off, bar_off,
        misc_off, total;
    __host__ __device__ TcLayout(int dk, int dv, int npad_max, int max_depth) {
        a_off = 0;                                               // H0 fp32 -> A bf16 hi,lo
        q_off = align_up(a_off + dk * dv * 4, 1024);             // q tiles, 128B-swizzled
        k_off = align_up(q_off + (dk / 64) * npad_max * 128, 1024);  // k rows [n][dk]
        v_off = align_up(k_off + npad_max * dk * 2, 1024);       // v rows [n][dv]
        x_off = align_up(v_off + npad_max * dv * 2, 16);         // lo-part exchange (dv = 64)
        w_off = align_up(x_off + (dv == 64 ? npad_max * 64 * 4 : 0), 16);
        eg_off = align_up(w_off + npad_max * max_depth * 4, 16);
        g_off = align_up(eg_off + npad_max * 4, 16);
        par_off = align_up(g_off + npad_max * 4, 16);
        dep_off = align_up(par_off + npad_max * 4, 16);
        bar_off = align_up(dep_off + npad_max * 4, 16);
        misc_off = bar_off + 32;
        total = align_up(misc_off + 16, 16) + 1024;  // + slack for 1024-byte base alignment
    }
};

struct TcParams {
    VerifyArgs a;
    int npad_max;
    int tmem_cols;
};

template <int DV>
__global__ void __launch_bounds__(kThreads, 1)
    verify_tc_scalar_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const TcParams P) {
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int dk = a.dk, H = a.H, md = a.max_depth;
    const TcLayout L(dk, DV, P.npad_max, md);
    float *sH0 = reinterpret_cast<float *>(smem + L.a_off);
    uint8_t *sA = smem + L.a_off;
    uint8_t *sQ = smem + L.q_off;
    const __nv_bfloat16 *sK = reinterpret_cast<const __nv_bfloat16 *>(smem + L.k_off);
    const __nv_bfloat16 *sV = reinterpret_cast<const __nv_bfloat16 *>(smem + L.v_off);
    float *sX = reinterpret_cast<float *>(smem + L.x_off);
    float *sW = reinterpret_cast<float *>(smem + L.w_off);
    float *sEG = reinterpret_cast<float *>(smem + L.eg_off);
    float *sG = reinterpret_cast<float *>(smem + L.g_off);
    int *sPar = reinterpret_cast<int *>(smem + L.par_off);
    int *sDep = reinterpret_cast<int *>(smem + L.dep_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sFlag = reinterpret_cast<int *>(smem + L.misc_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, b = unit / H, h = unit % H;
    const uint32_t bar_h0 = ptx::smem_addr(&bars[0]);
    const uint32_t bar_qkv = ptx::smem_addr(&bars[1]);
    const uint32_t bar_mma = ptx::smem_addr(&bars[2]);

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::mbar_init(bar_h0, 1);
        ptx::mbar_init(bar_qkv, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::fence_mbar_init();
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
        ptx::mbar_arrive_expect_tx(bar_h0, dk * DV * 4);
        ptx::bulk_g2s(ptx::smem_addr(sH0), a.H0 + (size_t)unit * dk * DV, dk * DV * 4, bar_h0);
    }

    int off = 0, n = 0;
    const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    if (!range_ok && tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
    const int npad = (n + 15) & ~15;
    const int slabs = dk / 64;
    const bool have_nodes = range_ok && n > 0;
    if (have_nodes && tid == 0) {
        const uint32_t tile = slabs * npad * 128;  // q or k bytes; v: npad * DV * 2
        ptx::mbar_arrive_expect_tx(bar_qkv, 2 * tile + npad * DV * 2);
        for (int r = 0; r < npad; r += 16) {
            for (int s = 0; s < slabs; ++s)
                ptx::tma_load_3d(ptx::smem_addr(sQ + s * P.npad_max * 128 + r * 128), &tm_q,
                                 s * 64, h, off + r, bar_qkv);
            ptx::tma_load_3d(ptx::smem_addr(sK) + r * dk * 2, &tm_k, 0, h, off + r, bar_qkv);
            ptx::tma_load_3d(ptx::smem_addr(sV) + r * DV * 2, &tm_v, 0, h, off + r, bar_qkv);
        }
    }
    ptx::grid_launch_dependents();

    // ---- tree checks and per-node decays while the copies fly
    bool ok = have_nodes;
    if (have_nodes) {
        for (int i = tid; i < n; i += kThreads) sG[i] = a.g[(size_t)(off + i) * H + h];
        ok = load_check_tree(a.parent, a.depth, off, n, md, sPar, sDep, sFlag);
        if (!ok) {
            for (int e = tid; e < n * DV; e += kThreads)
                a.out[((size_t)(off + e / DV) * H + h) * DV + e % DV] = 0.f;
            if (tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
        }
    }

    // ---- wait for the copies (always, so no copy outlives the CTA)
    bool landed = ptx::mbar_wait(bar_h0, 0, kWaitLimit);
    if (have_nodes) landed = landed && ptx::mbar_wait(bar_qkv, 0, kWaitLimit);
    const bool all_landed = __syncthreads_and(landed);
    if (!all_landed && tid == 0) report(a.status, TV_ERR_TIMEOUT);
    bool run = ok && all_landed;

    // ---- ancestor scores w_ij = e^{G_i - G_j} (q_i . k_j) and e^{G_i}, from shared memory
    if (run) {
        const int per_lane = dk / 32;               // 2 or 4 channels per lane
        const int c0 = lane * per_lane;             // within one 16-byte chunk
        for (int i = warp; i < n; i += kThreads / 32) {
            // q row i sits in a 128-byte-swizzled tile: chunk (c%64)/8 of row i moves to
            // chunk ((c%64)/8) ^ (i%8)
            const int slab = c0 / 64, cc = c0 % 64;
            const uint8_t *qrow = sQ + slab * P.npad_max * 128 + i * 128;
            const uint8_t *qp = qrow + ((((cc / 8) ^ (i & 7)) * 16) + (cc % 8) * 2);
            float qv[4];
            if (per_lane == 4) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(qp);
                const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
                const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
                qv[0] = __low2float(p0); qv[1] = __high2float(p0);
                qv[2] = __low2float(p1); qv[3] = __high2float(p1);
            } else {
                const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(qp);
                qv[0] = __low2float(p0); qv[1] = __high2float(p0);
                qv[2] = qv[3] = 0.f;
            }
            float s = 0.f;  // sum of g over the path nodes below the current ancestor
            int j = i, d = 0;
            while (j >= 0) {
                const __nv_bfloat16 *kr = sK + j * dk + c0;
                float part;
                if (per_lane == 4) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(kr);
                    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
                    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
                    part = qv[0] * __low2float(p0) + qv[1] * __high2float(p0) +
                           qv[2] * __low2float(p1) + qv[3] * __high2float(p1);
                } else {
                    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(kr);
                    part = qv[0] * __low2float(p0) + qv[1] * __high2float(p0);
                }
                part = warp_sum(part);
                if (lane == 0) sW[i * md + d] = expf(s) * part;
                s += sG[j];
                j = sPar[j];
                ++d;
            }
            if (lane == 0) sEG[i] = expf(s);
        }
    }

    // ---- split H0 (fp32, [dk][DV]) into bf16 hi/lo, rewritten as K-major A rows
    constexpr int kItems = DV * 128 / 8 / kThreads;  // (channel, 8-key) items per thread
    const int items = DV * (dk / 8);
    float hold[kItems][8];
    if (run) {
#pragma unroll
        for (int t = 0; t < kItems; ++t) {
            const int it = tid + t * kThreads;
            if (it < items) {
                const int c = it % DV, kq = it / DV;
#pragma unroll
                for (int e = 0; e < 8; ++e) hold[t][e] = sH0[(kq * 8 + e) * DV + c];
            }
        }
    }
    __syncthreads();
    const uint32_t sbo_a = dk * 16;  // bytes per 8-row group of A
    if (run) {
#pragma unroll
        for (int t = 0; t < kItems; ++t) {
            const int it = tid + t * kThreads;
            if (it < items) {
                const int c = it % DV, kq = it / DV;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x0 = hold[t][2 * e], x1 = hold[t][2 * e + 1];
                    const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                    const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
                    const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
                    hi[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                    lo[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                // hi part: rows 0..DV-1; lo part: rows DV..2DV-1 (stacked) for DV = 64,
                // or a second 128-row operand right after the first for DV = 128.
                const int r_hi = c, r_lo = DV + c;
                uint4 *ph = reinterpret_cast<uint4 *>(sA + (r_hi / 8) * sbo_a + kq * 128 + (r_hi % 8) * 16);
                uint4 *pl = reinterpret_cast<uint4 *>(sA + (r_lo / 8) * sbo_a + kq * 128 + (r_lo % 8) * 16);
                *ph = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *pl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();

    // ---- context term on the tensor core
    if (run && tid == 0) {
        const uint32_t idesc = ptx::idesc_bf16_f32(128, npad);
        const uint32_t a0 = ptx::smem_addr(sA), b0 = ptx::smem_addr(sQ);
        const int ksteps = dk / 16;
        const int passes = DV == 64 ? 1 : 2;  // DV = 128: hi operand, then lo operand
        for (int p = 0; p < passes; ++p) {
            const uint32_t abase = a0 + p * 16 * sbo_a;  // 128 rows further on
            for (int kk = 0; kk < ksteps; ++kk) {
                const uint64_t ad = ptx::desc_kmajor_noswizzle(abase + kk * 256, 128, sbo_a);
                const uint64_t bd = ptx::desc_kmajor_sw128(
                    b0 + (kk / 4) * P.npad_max * 128 + (kk % 4) * 32, 1024);
                ptx::mma_bf16(tmem, ad, bd, idesc, (p > 0 || kk > 0) ? 1u : 0u);
            }
        }
        ptx::mma_commit(bar_mma);
    }
    bool mma_ok = true;
    if (run) mma_ok = ptx::mbar_wait(bar_mma, 0, kWaitLimit);
    const bool all_mma = __syncthreads_and(mma_ok);
    if (run && !all_mma && tid == 0) report(a.status, TV_ERR_TIMEOUT);
    run = run && all_mma;
    ptx::tc_fence_after_sync();

    // ---- epilogue: lane = value channel, columns = nodes
    const int quad = warp & 3, half = warp >> 2;
    const int ncols_half = npad / 2;  // multiple of 8
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    if (DV == 64) {
        // quadrants 2,3 hold the lo part of channels 0..63: hand it over through smem
        if (run && quad >= 2) {
            const int c = 32 * (quad - 2) + lane;
            for (int col = half * ncols_half; col < (half + 1) * ncols_half; col += 8) {
                float vals[8];
                ptx::tmem_ld_x8(tq + col, vals);
#pragma unroll
                for (int e = 0; e < 8; ++e) sX[(col + e) * 64 + c] = vals[e];
            }
        }
        __syncthreads();
    }
    if (run && (DV == 128 || quad < 2)) {
        const int c = 32 * quad + lane;
        for (int col = half * ncols_half; col < (half + 1) * ncols_half; col += 8) {
            float vals[8];
            ptx::tmem_ld_x8(tq + col, vals);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = col + e;
                if (i >= n) break;
                float o = vals[e];
                if (DV == 64) o += sX[i * 64 + c];
                o *= sEG[i];
                int j = i, d = 0;
                while (j >= 0) {
                    o += sW[i * md + d] * __bfloat162float(sV[j * DV + c]);
                    j = sPar[j];
                    ++d;
                }
                a.out[((size_t)(off + i) * H + h) * DV + c] = o;
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int tmem_columns(int npad_max) {
    int c = 32;
    while (c < npad_max) c <<= 1;
    return c;
}

bool encode_rows(CUtensorMap *tm, const void *base, int width, int H, int T, int box_w,
                 CUtensorMapSwizzle swz) {
    // rows of `width` bf16 per (node, head): dims (width, H, T), one head per box
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * H};
    const cuuint32_t box[3] = {(cuuint32_t)box_w, 1, 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_fn()(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                       strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DV>
cudaError_t launch_dv(const VerifyArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv_;
    if (!encode_rows(&tq, a.q, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_rows(&tk, a.k, a.dk, a.H, a.T, a.dk, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_rows(&tv_, a.v, DV, a.H, a.T, DV, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    TcParams P;
    P.a = a;
    P.npad_max = (a.max_nodes + 15) & ~15;
    P.tmem_cols = tmem_columns(P.npad_max);
    const TcLayout L(a.dk, DV, P.npad_max, a.max_depth);
    size_t smem = L.total;
    auto kern = verify_tc_scalar_kernel<DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    // keep co-resident CTAs within the 512 tensor-memory columns of an SM
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    const int max_ctas = 512 / P.tmem_cols;
    if (per_sm > max_ctas) {
        // enlarge the request so that max_ctas + 1 blocks no longer fit on one SM
        int dev = 0, smem_sm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        size_t need = (size_t)smem_sm / (max_ctas + 1) + 1;
        if (need > smem) {
            smem = need;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * a.H));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv_, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool verify_tc_supported(const VerifyArgs &a) {
    return a.qkv_dtype == TV_BF16 && a.decay == TV_DECAY_SCALAR && (a.dk == 64 || a.dk == 128) &&
           (a.dv == 64 || a.dv == 128) && a.max_nodes <= kMaxNodes && encode_fn() != nullptr;
}

cudaError_t launch_verify_tc(const VerifyArgs &a, cudaStream_t s) {
    if (!verify_tc_supported(a)) return cudaErrorNotSupported;
    return a.dv == 64 ? launch_dv<64>(a, s) : launch_dv<128>(a, s);
}

}  // namespace tv
