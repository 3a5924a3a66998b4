// pack.cu -- one-time repack of the expert weights into the library layout (PackLayout).
//
// Fine-grained segmentation ([P1] "DeepSeekMoE 论文解读" (xxmr.cn), §两大核心策略) leaves every
// expert a SwiGLU FFN of intermediate width I. Two layout choices follow from the kernels:
//  - gate and up rows are interleaved in blocks of 16, so one accumulator tile of the gate/up GEMM
//    holds matching gate and up columns and the SwiGLU product is formed in its epilogue;
//  - the K_s shared experts, whose gates are all 1, are laid side by side as one expert of width
//    K_s*I: its down projection then sums the K_s expert outputs inside one GEMM.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Output row -> source, for a copy in 16-byte vectors by one warp per row.
//   region 0: gate/up routed  [N*2I rows of d]     region 1: gate/up shared [2*Ks*I rows of d]
//   region 2: down routed     [N*d rows of I]      region 3: down shared    [d rows of Ks*I]
__global__ void pack_kernel(Dims m, const char* __restrict__ wg, const char* __restrict__ wu,
                            const char* __restrict__ wd, char* __restrict__ out, PackLayout L) {
    const int region = blockIdx.y, es = m.elem();
    const size_t I = m.I, d = m.d, Ks = m.Ks, N = m.N;
    size_t n_rows, row_elems, out_base;
    switch (region) {
        case 0: n_rows = N * 2 * I; row_elems = d; out_base = L.gu_r; break;
        case 1: n_rows = Ks * 2 * I; row_elems = d; out_base = L.gu_s; break;
        case 2: n_rows = N * d; row_elems = I; out_base = L.dn_r; break;
        default: n_rows = Ks ? d : 0; row_elems = Ks * I; out_base = L.dn_s; break;
    }
    const int lane = threadIdx.x & 31;
    const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
    for (size_t r = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows;
         r += warps) {
        uint4* dst = reinterpret_cast<uint4*>(out + (out_base + r * row_elems) * es);
        const size_t vecs = row_elems * es / 16;
        if (region <= 1) {
            // packed row r: block b = r / 32 holds gate rows 16b..16b+15, then the same up rows
            const size_t e_rows = region == 0 ? 2 * I : 2 * Ks * I;
            const size_t e = r / e_rows, rr = r % e_rows, b = rr / 32, q = rr % 32;
            const size_t i = 16 * b + (q & 15);        // intermediate index within the expert
            const size_t src_row = region == 0 ? (Ks + e) * I + i : i;   // row of [E*I, d]
            const char* src = (q < 16 ? wg : wu) + src_row * d * es;
            for (size_t v = lane; v < vecs; v += 32)
                dst[v] = reinterpret_cast<const uint4*>(src)[v];
        } else if (region == 2) {
            const char* src = wd + (Ks * d * I + r * I) * es;   // routed experts follow the shared
            for (size_t v = lane; v < vecs; v += 32)
                dst[v] = reinterpret_cast<const uint4*>(src)[v];
        } else {
            // row n of the shared down projection: [W_down,0[n] | W_down,1[n] | ...]
            const size_t seg_vecs = I * es / 16;
            for (size_t v = lane; v < vecs; v += 32) {
                const size_t s = v / seg_vecs, w = v % seg_vecs;
                const char* src = wd + ((s * d + r) * I) * es;
                dst[v] = reinterpret_cast<const uint4*>(src)[w];
            }
        }
    }
}

}  // namespace

cudaError_t launch_pack(const Dims& m, const void* w_gate, const void* w_up, const void* w_down,
                        void* packed, cudaStream_t st) {
    const PackLayout L = pack_layout(m);
    dim3 grid(4 * sm_count(), 4);
    pack_kernel<<<grid, 256, 0, st>>>(m, static_cast<const char*>(w_gate),
                                      static_cast<const char*>(w_up),
                                      static_cast<const char*>(w_down),
                                      static_cast<char*>(packed), L);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
