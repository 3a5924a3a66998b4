// combine.cu -- gated combine with the residual, and the balance statistics.
//
// [P1] "DeepSeekMoE 论文解读" (xxmr.cn), §方法细节: h_t = sum_i g_{i,t} FFN_i(u_t) + u_t, with the
//      shared experts always active (gate 1); L_ExpBal = a1 sum_i f_i P_i; L_DevBal = a2 sum over
//      D groups of routed experts (one group per device).
// [P2] "【论文总结】MoE" (mickeyding.github.io), §2.3: f_i uses the factor N'/K' so the loss does not
//      depend on the expert count; §2.4: f'_i is the mean usage frequency of group i's experts and
//      P'_i the group's affinity (read here as the sum of P over the group).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <typename E> struct Vec;   // 16-byte vector of E
template <> struct Vec<float> {
    static constexpr int n = 4;
    __device__ static void load(const void* p, float* x) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    __device__ static void store(void* p, const float* x) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static void load(const void* p, float* x) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(h[q]);
            x[2 * q] = f.x;
            x[2 * q + 1] = f.y;
        }
    }
    __device__ static void store(void* p, const float* x) {
        uint4 v;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(x[2 * q], x[2 * q + 1]);
        *reinterpret_cast<uint4*>(p) = v;
    }
};

// One CTA per token; thread i owns 16-byte column vectors i, i + blockDim, ... of the row (one
// vector each for d <= 8 * blockDim in bf16). All 2 + KMAX row vectors of an iteration are loaded
// before any is used (slots k >= K' and bad rows read row 0 and are masked out), so every thread
// keeps that many loads in flight. fp32 accumulation in the fixed order u, shared sum, routed
// k = 0..K'-1.
template <typename E, int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(Dims m, const E* __restrict__ u,
                                                      const E* __restrict__ y_r,
                                                      const E* __restrict__ y_s,
                                                      const int* __restrict__ perm_slot,
                                                      const float* __restrict__ gate,
                                                      E* __restrict__ h, int* status,
                                                      long row_limit) {
    constexpr int VN = Vec<E>::n;
    const int t = blockIdx.x;
    const long TK = row_limit;   // rows of y_r
    int rows[KMAX];
    float g[KMAX];
    bool use[KMAX];
    bool bad = false;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        rows[k] = 0;
        g[k] = 0.f;
        use[k] = false;
        if (k < m.K) {
            const int r = perm_slot[(size_t)t * m.K + k];
            if (r < 0 || r >= TK) {
                bad = true;
            } else {
                rows[k] = r;
                g[k] = gate[(size_t)t * m.K + k];
                use[k] = true;
            }
        }
    }
    // the routing tables (written at least three launches earlier: the predecessor that this
    // kernel may overlap, the down GEMM, waited for them before it let this kernel start) and u
    // are read before the wait for that predecessor's outputs, y_r and y_s
    const int c0 = threadIdx.x * VN;
    uint4 raw_u0 = make_uint4(0u, 0u, 0u, 0u);
    if (c0 < m.d) raw_u0 = *reinterpret_cast<const uint4*>(u + (size_t)t * m.d + c0);
    pdl_wait();
    pdl_trigger();
    if (bad && threadIdx.x == 0) set_status(status, MOE_ERR_CORRUPT_INPUT);
    const bool shared = m.shared_active();
    for (int c = c0; c < m.d; c += blockDim.x * VN) {
        uint4 raw_u = c == c0 ? raw_u0 : *reinterpret_cast<const uint4*>(u + (size_t)t * m.d + c);
        uint4 raw_s = shared ? *reinterpret_cast<const uint4*>(y_s + (size_t)t * m.d + c) : raw_u;
        uint4 raw_r[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
            raw_r[k] = *reinterpret_cast<const uint4*>(y_r + (size_t)rows[k] * m.d + c);
        float acc[VN], y[VN];
        Vec<E>::load(&raw_u, acc);
        if (shared) {
            Vec<E>::load(&raw_s, y);
#pragma unroll
            for (int q = 0; q < VN; ++q) acc[q] += y[q];
        }
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (use[k]) {
                Vec<E>::load(&raw_r[k], y);
#pragma unroll
                for (int q = 0; q < VN; ++q) acc[q] = fmaf(g[k], y[q], acc[q]);
            }
        }
        Vec<E>::store(h + (size_t)t * m.d + c, acc);
    }
}

// One CTA; thread j handles expert j, thread 0 sums in expert order.
__global__ void balance_kernel(Dims m, const int* __restrict__ counts,
                               const float* __restrict__ psum, float* __restrict__ f_out,
                               float* __restrict__ P_out, float* __restrict__ losses) {
    __shared__ float f_s[kMaxRouted], P_s[kMaxRouted];
    const int N = m.N;
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        balance_fp(m, counts[j], psum[j], &f_s[j], &P_s[j]);
        f_out[j] = f_s[j];
        P_out[j] = P_s[j];
    }
    __syncthreads();
    if (threadIdx.x < 32) balance_losses_warp(m, f_s, P_s, losses, threadIdx.x);
}

}  // namespace

template <typename E, int KMAX>
void combine_t(const Dims& m, const void* u, const void* y_r, const void* y_s, const int* perm_slot,
               const float* gate, void* h, int* status, cudaStream_t st, long row_limit) {
    const int vecs = m.d * (int)sizeof(E) / 16;                 // 16-byte vectors per row
    const int threads = vecs >= 256 ? 256 : ((vecs + 31) / 32) * 32;
    launch_pdl(combine_kernel<E, KMAX>, dim3(m.T), dim3(threads), 0, st, m,
               static_cast<const E*>(u), static_cast<const E*>(y_r), static_cast<const E*>(y_s),
               perm_slot, gate, static_cast<E*>(h), status, row_limit);
}

cudaError_t launch_combine(const Dims& m, const void* u, const void* y_r, const void* y_s,
                           const int* perm_slot, const float* gate, void* h, int* status,
                           cudaStream_t st, long row_limit) {
    if (m.T == 0) return cudaSuccess;
    if (row_limit <= 0) row_limit = (long)m.T * m.K;
    if (m.dtype == MOE_DTYPE_F32) {
        if (m.K <= 4) combine_t<float, 4>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
        else if (m.K <= 8) combine_t<float, 8>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
        else combine_t<float, 16>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
    } else {
        using B = __nv_bfloat16;
        // the fine-grained configurations' K' (6, 12) get exact slot counts: no dummy row loads
        if (m.K <= 4) combine_t<B, 4>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
        else if (m.K <= 6) combine_t<B, 6>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
        else if (m.K <= 8) combine_t<B, 8>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
        else if (m.K <= 12) combine_t<B, 12>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
        else combine_t<B, 16>(m, u, y_r, y_s, perm_slot, gate, h, status, st, row_limit);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_balance(const Dims& m, const int* counts, const float* psum, float* f,
                          float* P, float* losses, cudaStream_t st) {
    balance_kernel<<<1, 256, 0, st>>>(m, counts, psum, f, P, losses);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
