// gemm_simt.cu -- grouped expert GEMMs for fp32 layers, on the CUDA cores in fp32.
//
// Same grouping and packed weights as the tensor-core path (groups.cuh, PackLayout): group 0 is
// the dense shared group, groups 1..N' the routed experts. Tiles are 64 rows x 64 output columns;
// each of 256 threads owns a 4 x 4 block. The gate/up kernel accumulates the gate and the up
// product of the same intermediate column side by side and writes silu(gate) * up directly.
#include "common.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int SB = 64;   // rows and output columns per tile
constexpr int SK = 16;   // K chunk staged in shared memory

struct SimtArgs {
    const float *a_r, *a_s;    // A matrices (row pitch = K extent)
    const float *b_r, *b_s;    // packed B rows (row pitch = K extent)
    int k_r, k_s;              // K extents
    int b_rows_per_expert;
    int n_out_r, n_out_s;      // output columns per group
    float *out_r, *out_s;      // outputs (row pitch = n_out)
    const int* offsets;
    GroupTiles gt;
};

// Packed row holding gate (up = false) or up (up = true) column i of a gate/up weight.
__device__ __forceinline__ int gu_row(int i, bool up) {
    return 32 * (i >> 4) + (i & 15) + (up ? 16 : 0);
}

template <bool GATEUP>
__global__ void __launch_bounds__(256) gemm_simt_kernel(SimtArgs a) {
    __shared__ int prefix[kMaxRouted + 2], rows_s[kMaxRouted + 2], row0_s[kMaxRouted + 2];
    __shared__ float As[SK][SB];
    __shared__ float Bs[SK][SB];
    __shared__ float Us[SK][SB];
    pdl_wait();
    pdl_trigger();
    build_tile_prefix<SB>(prefix, rows_s, row0_s, a.offsets, a.gt);
    const int total = prefix[a.gt.n_groups];
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TileInfo ti = decode_tile<SB>(t, prefix, rows_s, row0_s, a.gt);
        const bool sh = ti.group == 0;
        const float* A = sh ? a.a_s : a.a_r;
        const float* B = sh ? a.b_s : a.b_r + (size_t)(ti.group - 1) * a.b_rows_per_expert *
                                                    (size_t)a.k_r;
        const int K = sh ? a.k_s : a.k_r;
        const int n_out = sh ? a.n_out_s : a.n_out_r;
        float* out = sh ? a.out_s : a.out_r;
        const int r0 = ti.m_blk * SB, c0 = ti.n_blk * SB;
        float acc[4][4] = {}, accu[4][4] = {};
        for (int k0 = 0; k0 < K; k0 += SK) {
            // stage A [64 rows x 16] and B [64 cols x 16] (k-major in shared memory)
            for (int e = tid; e < SB * SK; e += 256) {
                const int r = e / SK, k = e % SK;
                const int gr = r0 + r;
                As[k][r] = gr < ti.m_rows ? A[(size_t)(ti.row0 + gr) * K + k0 + k] : 0.f;
                const int c = c0 + r;
                if (GATEUP) {
                    Bs[k][r] = c < n_out ? B[(size_t)gu_row(c, false) * K + k0 + k] : 0.f;
                    Us[k][r] = c < n_out ? B[(size_t)gu_row(c, true) * K + k0 + k] : 0.f;
                } else {
                    Bs[k][r] = c < n_out ? B[(size_t)c * K + k0 + k] : 0.f;
                }
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < SK; ++k) {
                float av[4], bv[4], uv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    av[i] = As[k][ty * 4 + i];
                    bv[i] = Bs[k][tx * 4 + i];
                    uv[i] = GATEUP ? Us[k][tx * 4 + i] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
                        if (GATEUP) accu[i][j] = fmaf(av[i], uv[j], accu[i][j]);
                    }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gr = r0 + ty * 4 + i;
            if (gr >= ti.m_rows) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = c0 + tx * 4 + j;
                if (c >= n_out) continue;
                const float v = GATEUP ? silu_f32(acc[i][j]) * accu[i][j] : acc[i][j];
                out[(size_t)(ti.row0 + gr) * n_out + c] = v;
            }
        }
    }
}

template <bool GATEUP>
cudaError_t run_simt(const Dims& m, SimtArgs a, cudaStream_t st) {
    a.gt.n_groups = 1 + m.N;
    a.gt.has_shared = m.shared_active();
    a.gt.T = m.T;
    a.gt.max_rows_r = m.T * m.K;
    a.gt.n_tiles_r = (a.n_out_r + SB - 1) / SB;
    a.gt.n_tiles_s = m.shared_active() ? (a.n_out_s + SB - 1) / SB : 0;
    a.gt.n_panel_s = 0;
    cudaError_t e = launch_pdl(gemm_simt_kernel<GATEUP>, dim3(4 * sm_count()), dim3(256), 0, st, a);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_gemms_simt(const Dims& m, const void* u, const void* x_perm,
                                     const void* packed, const int* offsets, void* act_r,
                                     void* act_s, void* y_r, void* y_s, cudaStream_t st,
                                     cudaEvent_t mid_event) {
    const PackLayout P = pack_layout(m);
    const float* pk = static_cast<const float*>(packed);
    const int KsI = m.Ks * m.I;
    SimtArgs gu{};
    gu.a_r = static_cast<const float*>(x_perm);
    gu.a_s = static_cast<const float*>(u);
    gu.b_r = pk + P.gu_r;
    gu.b_s = pk + P.gu_s;
    gu.k_r = gu.k_s = m.d;
    gu.b_rows_per_expert = 2 * m.I;
    gu.n_out_r = m.I;
    gu.n_out_s = KsI;
    gu.out_r = static_cast<float*>(act_r);
    gu.out_s = static_cast<float*>(act_s);
    gu.offsets = offsets;
    cudaError_t e = run_simt<true>(m, gu, st);
    if (e != cudaSuccess) return e;
    if (mid_event) cudaEventRecord(mid_event, st);
    SimtArgs dn{};
    dn.a_r = static_cast<const float*>(act_r);
    dn.a_s = static_cast<const float*>(act_s);
    dn.b_r = pk + P.dn_r;
    dn.b_s = pk + P.dn_s;
    dn.k_r = m.I;
    dn.k_s = KsI;
    dn.b_rows_per_expert = m.d;
    dn.n_out_r = dn.n_out_s = m.d;
    dn.out_r = static_cast<float*>(y_r);
    dn.out_s = static_cast<float*>(y_s);
    dn.offsets = offsets;
    return run_simt<false>(m, dn, st);
}

}  // namespace moe
