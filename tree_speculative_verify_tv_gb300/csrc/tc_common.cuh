// tc_common.cuh -- pieces shared by the tcgen05 verify kernels: the bf16 hi/lo
// split of fp32 state values, the 128-byte-swizzled operand layout, named
// barriers, and host helpers for tensor maps and tensor-memory sizing.
#pragma once

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc_ptx.cuh"
#include "tv_internal.cuh"

namespace tv {
namespace tcc {

constexpr long long kWaitLimit = 2000000000LL;  // ~1 s at 2 GHz

__host__ __device__ constexpr uint32_t align_up(uint32_t x, uint32_t a) {
    return (x + a - 1) / a * a;
}

constexpr int kChunkRows = 32;  // H0 key rows per streamed chunk
constexpr int kMaxChunks = 4;   // dk <= 128

__device__ __forceinline__ void load_bf16x(const __nv_bfloat16 *p, int cnt, float (&x)[4]) {
    if (cnt == 4) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(p);
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
        x[0] = __low2float(p0); x[1] = __high2float(p0);
        x[2] = __low2float(p1); x[3] = __high2float(p1);
    } else {
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(p);
        x[0] = __low2float(p0); x[1] = __high2float(p0);
        x[2] = x[3] = 0.f;
    }
}

// Byte offset of bf16 element (row, c) in a 128-byte-swizzled K-major tile:
// slab c/64 of `slab_bytes`, row of 128 bytes, 16-byte chunk (c%64)/8 XOR row%8.
__device__ __forceinline__ uint32_t swz_offset(int row, int c, uint32_t slab_bytes) {
    const int cc = c % 64;
    return (c / 64) * slab_bytes + row * 128 + ((((cc / 8) ^ (row & 7)) * 16) + (cc % 8) * 2);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// Split two floats into bf16 hi + lo parts: hi keeps the upper 16 bits (exact
// truncation), so x - hi is exact in fp32 and only lo is rounded (to nearest):
// |x - hi - lo| <= 2^-16 |x|.  Returns packed pairs (element 0 in the low half).
// The two remainders are formed by one packed fp32 subtraction (sub.f32x2).
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
    hi = __byte_perm(b0, b1, 0x7632);
    float r0, r1;
    asm("{\n\t.reg .b64 x, h, d;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 h, {%4, %5};\n\t"
        "sub.rn.f32x2 d, x, h;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(x0), "f"(x1), "r"(b0 & 0xFFFF0000u), "r"(b1 & 0xFFFF0000u));
    const __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// w_p *= q_i . k_j for every (node, ancestor) pair p = (i, j) of a request, pairs
// numbered node by node (sPairOff[n] of them; sPairNode[p] = i, sAnc[p] = j).  q is
// the 128-byte-swizzled bf16 B operand tile (slabs of 64 channels, `slab_bytes`
// apart), k dense bf16 rows of dk.  16 groups of 8 lanes (`grp` = this lane's
// group, the 128 threads of one warp group) take two pairs each per round, so the
// loads of a round are independent; the round count is uniform, so every lane of a
// warp takes each shuffle.  Lanes 4-7 of a group visit their two 16-byte pieces in
// the other order, which keeps each quarter-warp's loads of a k row and of the
// swizzled q row on distinct banks.
__device__ __forceinline__ void pair_scores(const uint8_t *sB, const __nv_bfloat16 *sK,
                                            const int *sPairOff, const uint8_t *sPairNode,
                                            const int *sAnc, float *sW, int n, int dk,
                                            uint32_t slab_bytes, int grp, int lane) {
    constexpr int kGroups = 16;
    const int npairs = sPairOff[n];
    const int sub = lane & 7;
    const int per = dk / 8;  // 16 or 8 key channels per lane, whole 16-byte chunks
    for (int base = 0; base < npairs; base += 2 * kGroups) {
        int pr[2], ii[2], jj[2];
        float acc[2];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            pr[x] = base + x * kGroups + grp;
            ii[x] = 0;
            jj[x] = 0;
            acc[x] = 0.f;
            if (pr[x] < npairs) {
                ii[x] = sPairNode[pr[x]];
                jj[x] = sAnc[pr[x]];
            }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            if (pr[x] < npairs) {
                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (u * 8 < per) {
                        const int uu = per == 16 ? ((u + (sub >> 2)) & 1) : u;
                        const int c = sub * per + uu * 8;
                        const uint4 qr =
                            *reinterpret_cast<const uint4 *>(sB + swz_offset(ii[x], c, slab_bytes));
                        const uint4 kr = *reinterpret_cast<const uint4 *>(sK + jj[x] * dk + c);
                        const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qr);
                        const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kr);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            p0 += __low2float(q2[e]) * __low2float(k2[e]);
                            p1 += __high2float(q2[e]) * __high2float(k2[e]);
                        }
                    }
                }
                acc[x] = p0 + p1;
            }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            float part = acc[x];
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            if (pr[x] < npairs && sub == 0) sW[pr[x]] *= part;
        }
    }
}

// Barrier among `count` threads and reduce: true iff `pred` holds in all of them.
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- host side

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

inline int tmem_columns(int npad_max) {
    int c = 32;
    while (c < npad_max) c <<= 1;
    return c;
}

inline bool encode_rows(CUtensorMap *tm, const void *base, CUtensorMapDataType dt, int esize, int width,
                        int H, int T, int box_w, CUtensorMapSwizzle swz) {
    // rows of `width` elements per (node, head): dims (width, H, T), one head per box
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)width * esize, (cuuint64_t)width * esize * H};
    const cuuint32_t box[3] = {(cuuint32_t)box_w, 1, 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_fn()(tm, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kSmemLimit = 227 * 1024;

// CTAs of `kern` resident on one SM at once: the least of what registers, shared memory
// (`smem` dynamic bytes) and tensor memory (`tmem_cols` columns of 512) allow.  The
// runtime's occupancy query knows nothing of tensor memory, and on this part it has
// reported fewer CTAs than the launch statistics show.
template <typename Kern>
cudaError_t resident_ctas(Kern kern, int threads, size_t smem, int tmem_cols, int &per_sm) {
    int dev = 0, smem_sm = 0, smem_rsv = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
            cudaSuccess)
        return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp
    const int by_regs = 65536 / (regs_warp * ((threads + 31) / 32));
    const int by_smem = smem_sm / (int)(smem + fa.sharedSizeBytes + smem_rsv);
    const int by_tmem = tmem_cols > 0 ? 512 / tmem_cols : 64;
    per_sm = std::max(1, std::min(std::min(by_regs, by_smem), by_tmem));
    return cudaSuccess;
}

}  // namespace tcc
}  // namespace tv
