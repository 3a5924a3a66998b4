// router.cu -- router of fp32 layers on the CUDA cores (bf16 layers: router_tc.cu).
//
// [P1] "DeepSeekMoE 论文解读" (xxmr.cn), §方法细节: gates g_{i,t} come from Topk({s_{j,t}}, mK);
//      the K_s shared experts are always active, so routing ranks only the N' routed experts.
// [P2] "【论文总结】MoE" (mickeyding.github.io), §2.2: s_{j,t} scores token t against the learnable
//      centroid e_j; §2.3: f_i counts selections, P_i averages s over the T tokens.
//
// Ranking uses the logits z = u.e + b: softmax is strictly increasing in z, so the K' largest z are
// the K' largest s, and equal z give equal s. Ties go to the lower expert index.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRouterThreads = 256;

// Top-KMAX insertion list, kept sorted by value descending. Candidates arrive in ascending
// expert index, and a candidate displaces an entry only if strictly larger, so equal values
// keep the lower index ahead.
template <int KMAX>
struct TopList {
    float v[KMAX];
    int i[KMAX];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int q = 0; q < KMAX; ++q) {
            v[q] = -INFINITY;
            i[q] = -1;
        }
    }
    __device__ __forceinline__ void push(float x, int j) {
        if (!(x > v[KMAX - 1])) return;
#pragma unroll
        for (int q = KMAX - 1; q > 0; --q) {
            if (x > v[q]) {
                if (x > v[q - 1]) {
                    v[q] = v[q - 1];
                    i[q] = i[q - 1];
                } else {
                    v[q] = x;
                    i[q] = j;
                }
            }
        }
        if (x > v[0]) {
            v[0] = x;
            i[0] = j;
        }
    }
};

template <typename E> struct Pair;
template <> struct Pair<float> {
    using V = float2;
    __device__ static float2 f2(V x) { return x; }
};

// One CTA per 128-token tile. Phase 1: each warp computes the logits of its tokens (lanes split
// the model dimension, 4 experts per pass, warp-shuffle reduction) into shared memory.
// Phase 2: one thread per token turns its logit row into affinities, top-k and gates.
// Phase 3: one thread per expert sums the tile's affinities in token order.
template <typename E, int KMAX>
__global__ void __launch_bounds__(kRouterThreads)
router_simt_kernel(const E* __restrict__ u, const E* __restrict__ cent,
                   const float* __restrict__ bias, Dims m, int* __restrict__ topk_idx,
                   float* __restrict__ topk_gate, int* __restrict__ tile_counts,
                   float* __restrict__ tile_psum, int* status) {
    extern __shared__ float z_s[];                 // [kRouteTile][N]
    __shared__ int hist[kMaxRouted];
    using V = typename Pair<E>::V;
    const int N = m.N, d = m.d, K = m.K;
    const int tile = blockIdx.x, t0 = tile * kRouteTile;
    const int n_tok = min(kRouteTile, m.T - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    for (int j = threadIdx.x; j < N; j += blockDim.x) hist[j] = 0;

    for (int tl = warp; tl < n_tok; tl += kRouterThreads / 32) {
        const V* ur = reinterpret_cast<const V*>(u + (size_t)(t0 + tl) * d);
        for (int j0 = 0; j0 < N; j0 += 4) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c = lane; c < d / 2; c += 32) {
                const float2 x = Pair<E>::f2(ur[c]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (j0 + q < N) {
                        const float2 w = Pair<E>::f2(
                            reinterpret_cast<const V*>(cent + (size_t)(j0 + q) * d)[c]);
                        acc[q] = fmaf(x.x, w.x, acc[q]);
                        acc[q] = fmaf(x.y, w.y, acc[q]);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float a = acc[q];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                if (lane == 0 && j0 + q < N)
                    z_s[tl * N + j0 + q] = a + (bias ? bias[j0 + q] : 0.f);
            }
        }
    }
    __syncthreads();

    if (threadIdx.x < n_tok) {
        const int tl = threadIdx.x, t = t0 + tl;
        float* z = z_s + tl * N;
        float zmax = -INFINITY;
        for (int j = 0; j < N; ++j) zmax = fmaxf(zmax, z[j]);
        TopList<KMAX> top;
        top.init();
        float sum = 0.f;
        for (int j = 0; j < N; ++j) {
            top.push(z[j], j);
            sum += expf(z[j] - zmax);
        }
        const float inv = 1.0f / sum;
        for (int j = 0; j < N; ++j) z[j] = expf(z[j] - zmax) * inv;   // z row now holds s
        const int q0 = m.skip;   // chosen ranks: q0 .. q0+K'-1
        float gsum = 0.f;
#pragma unroll
        for (int q = 0; q < KMAX; ++q)
            if (q >= q0 && q < q0 + K) gsum += expf(top.v[q] - zmax) * inv;
        bool bad = !(zmax < INFINITY);
#pragma unroll
        for (int q = 0; q < KMAX; ++q) {
            if (q >= q0 && q < q0 + K) {
                int j = top.i[q];
                if (j < 0) { bad = true; j = 0; }
                const float s = expf(top.v[q] - zmax) * inv;
                topk_idx[(size_t)t * K + q - q0] = j;
                topk_gate[(size_t)t * K + q - q0] = m.renorm ? s / gsum : s;
                atomicAdd(&hist[j], 1);
            }
        }
        if (bad) set_status(status, MOE_ERR_CORRUPT_INPUT);
    }
    __syncthreads();

    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        float acc = 0.f;
        for (int tl = 0; tl < n_tok; ++tl) acc += z_s[tl * N + j];
        tile_psum[(size_t)j * gridDim.x + tile] = acc;
        tile_counts[(size_t)j * gridDim.x + tile] = hist[j];
    }
}

template <typename E, int KMAX>
cudaError_t launch_router_t(const Dims& m, const void* u, const void* cent, const float* bias,
                            int* idx, float* gate, int* tc, float* tp, int* status,
                            cudaStream_t st) {
    const int n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    const size_t smem = (size_t)kRouteTile * m.N * sizeof(float);
    auto kern = router_simt_kernel<E, KMAX>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(n_tiles), dim3(kRouterThreads), smem, st, static_cast<const E*>(u),
                   static_cast<const E*>(cent), bias, m, idx, gate, tc, tp, status);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const Dims& m, const void* u, const void* centroids, const float* bias,
                          int* topk_idx, float* topk_gate, int* tile_counts, float* tile_psum,
                          int* status, cudaStream_t st) {
    if (m.T == 0) return cudaSuccess;
    if (m.dtype == MOE_DTYPE_BF16)
        return launch_router_tc(m, u, centroids, bias, topk_idx, topk_gate, tile_counts,
                                tile_psum, status, st);
    return m.skip + m.K <= 8 ? launch_router_t<float, 8>(m, u, centroids, bias, topk_idx, topk_gate,
                                                tile_counts, tile_psum, status, st)
                    : launch_router_t<float, 16>(m, u, centroids, bias, topk_idx, topk_gate,
                                                 tile_counts, tile_psum, status, st);
}

}  // namespace moe
