// verify_serial.cu -- the naive serial tree verification on the GPU, as a
// baseline for the tree closed form.
//
// Bole summary page: the naive way verifies a linear-recurrence layer over a draft
// tree by walking the nodes one after another and keeping a full state matrix for
// every node (the per-node states the closed form avoids, "Core techniques" §1-§2):
//   S_i = diag(exp g_i) S_parent(i) + k_i v_i^T   (S_parent = H0 at the context)
//   o_i = S_i^T q_i
// Here the (request, head) units run in parallel, one CTA each, and inside a unit
// the nodes are processed in index order (parents precede children).  Every S_i is
// written to the caller's workspace [B*H][max_nodes][dk][dv] fp32 and re-read as
// the parent of later nodes; H0 is only read.
//
// Per node, each of 256 threads updates its share of the dk x dv state as float4s
// (dk*dv/1024 float4 each, dv >= 4) and accumulates S_i^T q_i over its rows; the
// column sums are reduced through shared memory.
#include "tv_internal.cuh"

// Scratch of tv_verify_serial_static: the per-node states of problems that need at
// most TV_SERIAL_STATIC_BYTES.  One copy lives on every device that loads the
// library; host code only uses its name to look up that device address.
static __device__ __align__(256) float g_serial_states[TV_SERIAL_STATIC_BYTES / sizeof(float)];

namespace tv {
namespace {

constexpr int kThreadsS = 256;

template <typename E, bool DIAG>
__global__ void __launch_bounds__(kThreadsS) verify_serial_kernel(VerifyArgs a, float *ws) {
    __shared__ int s_par[kMaxNodes];
    __shared__ int s_dep[kMaxNodes];
    __shared__ int s_flag;
    extern __shared__ float s_dyn[];  // q_i, k_i, decay_i [dk] each; v_i [dv]; [row groups][dv]
    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit % a.H;
    const int tid = threadIdx.x;
    const int dk = a.dk, dv = a.dv, H = a.H;
    const E *q = static_cast<const E *>(a.q);
    const E *k = static_cast<const E *>(a.k);
    const E *v = static_cast<const E *>(a.v);
    float *sq = s_dyn, *sk = sq + dk, *se = sk + dk, *sv = se + dk;
    float *spart = sv + dv;  // [row groups][dv]

    pdl_wait();
    pdl_launch_next();
    int off, n;
    if (!request_range(a.node_offsets, b, a.T, a.max_nodes, off, n)) {
        if (tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
        return;
    }
    if (!load_check_tree(a.parent, a.depth, off, n, a.max_depth, s_par, s_dep, &s_flag)) {
        if (tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
        for (int e = tid; e < n * dv; e += kThreadsS)
            a.out[((size_t)(off + e / dv) * H + h) * dv + e % dv] = 0.f;
        return;
    }

    // thread layout over the state: c4 = column quad, rg = row group
    const int c4n = dv / 4;
    const int groups = kThreadsS / c4n;  // row groups (dv <= 1024)
    const int c4 = tid % c4n, rg = tid / c4n;
    const bool active = rg < groups;
    const size_t sz = (size_t)dk * dv;
    const float *H0u = a.H0 + (size_t)unit * sz;
    float *wsu = ws + (size_t)unit * a.max_nodes * sz;

    for (int i = 0; i < n; ++i) {
        const size_t row = (size_t)(off + i) * H + h;
        for (int r = tid; r < dk; r += kThreadsS) {
            sq[r] = ldg_f(q, row * dk + r);
            sk[r] = ldg_f(k, row * dk + r);
            se[r] = expf(DIAG ? a.g[row * dk + r] : a.g[row]);
        }
        for (int c = tid; c < dv; c += kThreadsS) sv[c] = ldg_f(v, row * dv + c);
        __syncthreads();
        const int p = s_par[i];
        const float *src = p < 0 ? H0u : wsu + (size_t)p * sz;
        float *dst = wsu + (size_t)i * sz;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active) {
            const float4 vv = *reinterpret_cast<const float4 *>(sv + 4 * c4);
            for (int r = rg; r < dk; r += groups) {
                float4 s = *reinterpret_cast<const float4 *>(src + (size_t)r * dv + 4 * c4);
                const float e = se[r], kr = sk[r], qr = sq[r];
                s.x = e * s.x + kr * vv.x;
                s.y = e * s.y + kr * vv.y;
                s.z = e * s.z + kr * vv.z;
                s.w = e * s.w + kr * vv.w;
                *reinterpret_cast<float4 *>(dst + (size_t)r * dv + 4 * c4) = s;
                acc.x += qr * s.x;
                acc.y += qr * s.y;
                acc.z += qr * s.z;
                acc.w += qr * s.w;
            }
            *reinterpret_cast<float4 *>(spart + rg * dv + 4 * c4) = acc;
        }
        __syncthreads();  // partial sums ready; S_i written before a child reads it
        for (int c = tid; c < dv; c += kThreadsS) {
            float o = 0.f;
            for (int g2 = 0; g2 < groups; ++g2) o += spart[g2 * dv + c];
            a.out[row * dv + c] = o;
        }
        __syncthreads();  // shared vectors are rewritten for the next node
    }
}

template <typename E, bool DIAG>
cudaError_t launch_typed(const VerifyArgs &a, float *ws, cudaStream_t s) {
    const int groups = kThreadsS / (a.dv / 4);
    const size_t smem = ((size_t)3 * a.dk + a.dv + (size_t)groups * a.dv) * sizeof(float);
    const cudaError_t attr = configure_smem_once(verify_serial_kernel<E, DIAG>, false);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(verify_serial_kernel<E, DIAG>, dim3((unsigned)(a.B * a.H)),
                      dim3(kThreadsS), smem, s, a, ws);
}

}  // namespace

size_t verify_serial_workspace_bytes(const VerifyArgs &a) {
    return (size_t)a.B * a.H * a.max_nodes * a.dk * a.dv * sizeof(float);
}

namespace {

// Device address of g_serial_states on the current device.  It is looked up on
// every call (cheap once the module is loaded), so the address is never stale, for
// instance after the caller reset the device.
cudaError_t static_states(float **ptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_serial_states);
    if (e != cudaSuccess) return e;
    *ptr = static_cast<float *>(p);
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_verify_serial(const VerifyArgs &a, float *ws, cudaStream_t s) {
    const bool diag = a.decay == TV_DECAY_DIAG;
    if (a.qkv_dtype == TV_BF16)
        return diag ? launch_typed<__nv_bfloat16, true>(a, ws, s)
                    : launch_typed<__nv_bfloat16, false>(a, ws, s);
    return diag ? launch_typed<float, true>(a, ws, s) : launch_typed<float, false>(a, ws, s);
}

cudaError_t launch_verify_serial_static(const VerifyArgs &a, cudaStream_t s) {
    if (verify_serial_workspace_bytes(a) > TV_SERIAL_STATIC_BYTES) return cudaErrorInvalidValue;
    float *ws = nullptr;
    const cudaError_t e = static_states(&ws);
    if (e != cudaSuccess) return e;
    return launch_verify_serial(a, ws, s);
}

}  // namespace tv
