// backward.cu -- elementwise and gather/scatter kernels of the layer backward (bf16 layers).
//
// Objective: sum_t dh_t . h_t + L_ExpBal + L_DevBal, with the expert selection and the counts
// held fixed ([P1] "DeepSeekMoE 论文解读" (xxmr.cn), §方法细节: h_t = sum_i g_{i,t} FFN_i(u_t) + u_t,
// f_i a selection frequency, P_i a mean affinity; [P2] "【论文总结】MoE" §2.3, §2.4).
//
// Routed rows live in padded per-expert segments: expert j owns rows poff[j] .. poff[j+1]-1,
// poff[j] a multiple of 64, its count_j real rows first and zero rows after them, so the weight
// gradients can reduce over whole 64-row blocks.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Transposed copies of the expert weights for the input-gradient GEMMs (PackBwdLayout).
//   region 0: WdT_r [N, I, d]  (W_down,e^T)       region 1: WdT_s [Ks*I, d]
//   region 2: WguT_r [N, d, 2I] (packed gate/up^T) region 3: WguT_s [d, 2*Ks*I]
// One thread per output element (a one-time repack).
__global__ void pack_bwd_kernel(Dims m, const __nv_bfloat16* __restrict__ wg,
                                const __nv_bfloat16* __restrict__ wu,
                                const __nv_bfloat16* __restrict__ wd,
                                __nv_bfloat16* __restrict__ out, PackBwdLayout L) {
    const size_t I = m.I, d = m.d, Ks = m.Ks, N = m.N;
    const int region = blockIdx.y;
    size_t n, base;
    switch (region) {
        case 0: n = N * I * d; base = L.wdT_r; break;
        case 1: n = Ks * I * d; base = L.wdT_s; break;
        case 2: n = N * d * 2 * I; base = L.wguT_r; break;
        default: n = d * 2 * Ks * I; base = L.wguT_s; break;
    }
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < n;
         o += (size_t)gridDim.x * blockDim.x) {
        __nv_bfloat16 v;
        if (region == 0) {          // WdT_r[e][i][c] = W_down[K_s + e][c][i]
            const size_t e = o / (I * d), r = o % (I * d), i = r / d, c = r % d;
            v = wd[((Ks + e) * d + c) * I + i];
        } else if (region == 1) {   // WdT_s[s*I + i][c] = W_down[s][c][i]
            const size_t gi = o / d, c = o % d, se = gi / I, i = gi % I;
            v = wd[(se * d + c) * I + i];
        } else {
            // WguT[e][c][p] = packed gate/up row p (gate 16b+q for q<16, up otherwise), column c
            const size_t P = region == 2 ? 2 * I : 2 * Ks * I;
            const size_t e = o / (d * P), r = o % (d * P), c = r / P, p = r % P;
            const size_t b = p / 32, q = p % 32, i = 16 * b + (q & 15);   // intermediate index
            const size_t row = region == 2 ? (Ks + e) * I + i : i;        // row of [E*I, d]
            v = (q < 16 ? wg : wu)[row * d + c];
        }
        out[base + o] = v;
    }
}

// Zero rows of the padded segments: rows poff[j] + count[j] .. poff[j+1]-1 of each listed buffer
// (row width `width` bf16). One CTA per expert.
__global__ void zero_pad_rows_kernel(int N, const int* __restrict__ poff,
                                     const int* __restrict__ counts, __nv_bfloat16* b0,
                                     __nv_bfloat16* b1, int width) {
    pdl_wait();
    pdl_trigger();
    const int j = blockIdx.x;
    const int r0 = poff[j] + counts[j], r1 = poff[j + 1];
    const size_t vecs = (size_t)(r1 - r0) * width / 8;   // 16-byte vectors
    uint4 z = make_uint4(0, 0, 0, 0);
    for (size_t v = threadIdx.x; v < vecs; v += blockDim.x) {
        reinterpret_cast<uint4*>(b0 + (size_t)r0 * width)[v] = z;
        if (b1) reinterpret_cast<uint4*>(b1 + (size_t)r0 * width)[v] = z;
    }
}

// Combine backward, one CTA per token: d_y[row_k] = g_k * dh_t (bf16) and
// dgate[t, k] = dh_t . y[row_k] (fp32, block reduction in a fixed order).
__global__ void __launch_bounds__(256) combine_bwd_kernel(Dims m, const __nv_bfloat16* __restrict__ dh,
                                                        const __nv_bfloat16* __restrict__ y_r,
                                                        const int* __restrict__ perm_slot,
                                                        const float* __restrict__ gate,
                                                        __nv_bfloat16* __restrict__ d_y,
                                                        float* __restrict__ dgate) {
    __shared__ float red[kMaxTopK][8];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const __nv_bfloat16* dht = dh + (size_t)t * m.d;
    for (int k = 0; k < m.K; ++k) {
        const int row = perm_slot[(size_t)t * m.K + k];
        const float g = gate[(size_t)t * m.K + k];
        const __nv_bfloat16* yr = y_r + (size_t)row * m.d;
        __nv_bfloat16* dyr = d_y + (size_t)row * m.d;
        float dot = 0.f;
        for (int c = threadIdx.x * 8; c < m.d; c += blockDim.x * 8) {
            const uint4 hv = *reinterpret_cast<const uint4*>(dht + c);
            const uint4 yv = *reinterpret_cast<const uint4*>(yr + c);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hv);
            const __nv_bfloat162* y2 = reinterpret_cast<const __nv_bfloat162*>(&yv);
            uint4 ov;
            __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&ov);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 hf = __bfloat1622float2(h2[q]), yf = __bfloat1622float2(y2[q]);
                dot = fmaf(hf.x, yf.x, dot);
                dot = fmaf(hf.y, yf.y, dot);
                o2[q] = __floats2bfloat162_rn(g * hf.x, g * hf.y);
            }
            *reinterpret_cast<uint4*>(dyr + c) = ov;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) red[k][warp] = dot;
    }
    __syncthreads();
    if (threadIdx.x < m.K) {
        float s = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[threadIdx.x][w];
        dgate[(size_t)t * m.K + threadIdx.x] = s;
    }
}

// du_t = dh_t + d_x_shared[t] + d_u_router[t] + sum_k d_x[perm_slot[t, k]] (fp32 out, fixed
// order). One CTA per token, 8 columns per thread per step, all 3 + KMAX row loads issued before
// any is summed (slots k >= K' load row 0 and are skipped).
template <int KMAX>
__global__ void __launch_bounds__(256) du_final_kernel(Dims m, const __nv_bfloat16* __restrict__ dh,
                                                     const __nv_bfloat16* __restrict__ dx_s,
                                                     const __nv_bfloat16* __restrict__ du_r,
                                                     const __nv_bfloat16* __restrict__ dx,
                                                     const int* __restrict__ perm_slot,
                                                     float* __restrict__ du) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    int rows[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) rows[k] = k < m.K ? perm_slot[(size_t)t * m.K + k] : 0;
    const bool shared = m.shared_active();
    for (int c = threadIdx.x * 8; c < m.d; c += blockDim.x * 8) {
        const size_t o = (size_t)t * m.d + c;
        uint4 raw[3 + KMAX];
        raw[0] = *reinterpret_cast<const uint4*>(dh + o);
        raw[1] = shared ? *reinterpret_cast<const uint4*>(dx_s + o) : make_uint4(0, 0, 0, 0);
        raw[2] = *reinterpret_cast<const uint4*>(du_r + o);
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
            raw[3 + k] = *reinterpret_cast<const uint4*>(dx + (size_t)rows[k] * m.d + c);
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
        for (int k = 0; k < 3 + KMAX; ++k) {
            if (k < 3 + m.K) {
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __bfloat1622float2(h2[q]);
                    acc[2 * q] += f.x;
                    acc[2 * q + 1] += f.y;
                }
            }
        }
        float4* out = reinterpret_cast<float4*>(du + o);
        out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// Router transposed centroids: eT [d, n_pad] (bf16, zero for j >= N') for d_u = dz e.
__global__ void transpose_centroids_kernel(int N, int n_pad, int d,
                                           const __nv_bfloat16* __restrict__ e,
                                           __nv_bfloat16* __restrict__ eT) {
    pdl_wait();
    pdl_trigger();
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < (size_t)d * n_pad;
         o += (size_t)gridDim.x * blockDim.x) {
        const size_t c = o / n_pad, j = o % n_pad;
        eT[o] = j < (size_t)N ? e[j * d + c] : __float2bfloat16_rn(0.f);
    }
}

// d_bias[j] = sum over tiles of the per-tile column sums of dz (tile order). One warp per expert.
__global__ void dbias_reduce_kernel(int N, int n_tiles, const float* __restrict__ tile_dz,
                                    float* __restrict__ d_bias) {
    pdl_wait();
    pdl_trigger();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= N) return;
    float s = 0.f;
    for (int t = lane; t < n_tiles; t += 32) s += tile_dz[(size_t)warp * n_tiles + t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) d_bias[warp] = s;
}

}  // namespace

cudaError_t launch_pack_bwd(const Dims& m, const void* w_gate, const void* w_up,
                            const void* w_down, void* packed_bwd, cudaStream_t st) {
    pack_bwd_kernel<<<dim3(4 * sm_count(), 4), 256, 0, st>>>(
        m, static_cast<const __nv_bfloat16*>(w_gate), static_cast<const __nv_bfloat16*>(w_up),
        static_cast<const __nv_bfloat16*>(w_down), static_cast<__nv_bfloat16*>(packed_bwd),
        pack_bwd_layout(m));
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_zero_pad_rows(const Dims& m, const int* poff, const int* counts, void* b0,
                                 void* b1, int width, cudaStream_t st) {
    cudaError_t e = launch_pdl(zero_pad_rows_kernel, dim3(m.N), dim3(256), 0, st, m.N, poff,
                               counts, static_cast<__nv_bfloat16*>(b0),
                               static_cast<__nv_bfloat16*>(b1), width);
    note_launches(1);
    return e;
}

cudaError_t launch_combine_bwd(const Dims& m, const void* dh, const void* y_r,
                               const int* perm_slot, const float* gate, void* d_y, float* dgate,
                               cudaStream_t st) {
    if (m.T == 0) return cudaSuccess;
    const int threads = std::min(256, std::max(32, ((m.d / 8 + 31) / 32) * 32));
    cudaError_t e = launch_pdl(combine_bwd_kernel, dim3(m.T), dim3(threads), 0, st, m,
                               static_cast<const __nv_bfloat16*>(dh),
                               static_cast<const __nv_bfloat16*>(y_r), perm_slot, gate,
                               static_cast<__nv_bfloat16*>(d_y), dgate);
    note_launches(1);
    return e;
}

cudaError_t launch_du_final(const Dims& m, const void* dh, const void* dx_s, const void* du_r,
                            const void* dx, const int* perm_slot, float* du, cudaStream_t st) {
    if (m.T == 0) return cudaSuccess;
    const int threads = std::min(256, std::max(32, ((m.d / 8 + 31) / 32) * 32));
    auto kern = m.K <= 4 ? du_final_kernel<4> : (m.K <= 8 ? du_final_kernel<8> : du_final_kernel<16>);
    cudaError_t e = launch_pdl(kern, dim3(m.T), dim3(threads), 0, st, m,
                               static_cast<const __nv_bfloat16*>(dh),
                               static_cast<const __nv_bfloat16*>(dx_s),
                               static_cast<const __nv_bfloat16*>(du_r),
                               static_cast<const __nv_bfloat16*>(dx), perm_slot, du);
    note_launches(1);
    return e;
}

cudaError_t launch_transpose_centroids(const Dims& m, int n_pad, const void* e, void* eT,
                                       cudaStream_t st) {
    const size_t n = (size_t)m.d * n_pad;
    const int blocks = (int)std::min<size_t>((n + 255) / 256, (size_t)sm_count() * 8);
    cudaError_t err = launch_pdl(transpose_centroids_kernel, dim3(blocks), dim3(256), 0, st, m.N,
                                 n_pad, m.d, static_cast<const __nv_bfloat16*>(e),
                                 static_cast<__nv_bfloat16*>(eT));
    note_launches(1);
    return err;
}

cudaError_t launch_dbias_reduce(int N, int n_tiles, const float* tile_dz, float* d_bias,
                                cudaStream_t st) {
    cudaError_t e = launch_pdl(dbias_reduce_kernel, dim3((N * 32 + 255) / 256), dim3(256), 0, st,
                               N, n_tiles, tile_dz, d_bias);
    note_launches(1);
    return e;
}

}  // namespace moe
