// permute.cu -- dispatch of the routed assignments: per-expert histogram, offsets, a stable
// counting-sort permutation (expert-major, tokens ascending inside an expert) and the gather of
// token rows into that order.
//
// The pages activate only the chosen experts per token ([P1] "DeepSeekMoE 论文解读" (xxmr.cn),
// §方法细节), which is what makes the expert GEMMs grouped: expert j works on the contiguous rows
// offsets[j] .. offsets[j+1]-1 of the permuted token matrix.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Histogram of one 128-token tile of topk_idx. Out-of-range ids are skipped and flagged.
__global__ void tile_hist_kernel(Dims m, const int* __restrict__ topk_idx,
                                 int* __restrict__ tile_counts, int* status) {
    __shared__ int hist[kMaxRouted];
    const int tile = blockIdx.x, t0 = tile * kRouteTile;
    const int n = min(kRouteTile, m.T - t0) * m.K;
    for (int j = threadIdx.x; j < m.N; j += blockDim.x) hist[j] = 0;
    __syncthreads();
    const int* idx = topk_idx + (size_t)t0 * m.K;
    bool bad = false;
    for (int a = threadIdx.x; a < n; a += blockDim.x) {
        const int j = idx[a];
        if (j >= 0 && j < m.N) atomicAdd(&hist[j], 1);
        else bad = true;
    }
    if (bad) set_status(status, MOE_ERR_CORRUPT_INPUT);
    __syncthreads();
    for (int j = threadIdx.x; j < m.N; j += blockDim.x)
        tile_counts[(size_t)tile * m.N + j] = hist[j];
}

// One CTA: per expert, the running base over tiles (token order), the total, the check against
// the caller's counts, then offsets by an exclusive scan over experts.
__global__ void perm_scan_kernel(Dims m, int n_tiles, const int* __restrict__ tile_counts,
                                 const int* __restrict__ counts, int* __restrict__ offsets,
                                 int* __restrict__ tile_base, int* status) {
    __shared__ int total[kMaxRouted];
    __shared__ int off[kMaxRouted + 1];
    const int N = m.N;
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        int run = 0;
        for (int tile = 0; tile < n_tiles; ++tile) {
            tile_base[(size_t)tile * N + j] = run;
            run += tile_counts[(size_t)tile * N + j];
        }
        total[j] = run;
        if (counts && counts[j] != run) set_status(status, MOE_ERR_CORRUPT_INPUT);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int j = 0; j < N; ++j) {
            off[j] = acc;
            acc += total[j];
        }
        off[N] = acc;
    }
    __syncthreads();
    for (int j = threadIdx.x; j <= N; j += blockDim.x) offsets[j] = off[j];
    for (int j = threadIdx.x; j < N; j += blockDim.x)
        for (int tile = 0; tile < n_tiles; ++tile) tile_base[(size_t)tile * N + j] += off[j];
}

// One CTA per tile: thread j walks the tile's assignments in (token, slot) order and hands out
// consecutive rows of expert j, which keeps tokens ascending inside every expert.
__global__ void perm_scatter_kernel(Dims m, const int* __restrict__ topk_idx,
                                    const int* __restrict__ tile_base, int* __restrict__ perm_token,
                                    int* __restrict__ perm_slot) {
    __shared__ int idx_s[kRouteTile * kMaxTopK];
    const int tile = blockIdx.x, t0 = tile * kRouteTile, K = m.K;
    const int n = min(kRouteTile, m.T - t0) * K;
    for (int a = threadIdx.x; a < n; a += blockDim.x) {
        const int j = topk_idx[(size_t)t0 * K + a];
        idx_s[a] = j;
        if (j < 0 || j >= m.N) perm_slot[(size_t)t0 * K + a] = -1;   // flagged by the histogram
    }
    __syncthreads();
    for (int j = threadIdx.x; j < m.N; j += blockDim.x) {
        int row = tile_base[(size_t)tile * m.N + j];
        for (int a = 0; a < n; ++a) {
            if (idx_s[a] == j) {
                perm_token[row] = t0 + a / K;
                perm_slot[(size_t)t0 * K + a] = row;
                ++row;
            }
        }
    }
}

// One warp per token: the row is read once (16-byte vectors) and written to its K' rows.
__global__ void gather_kernel(Dims m, const uint4* __restrict__ u, const int* __restrict__ perm_slot,
                              uint4* __restrict__ x_perm, int* status) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= m.T) return;
    const int vec_per_row = m.d * m.elem() / 16;
    const long TK = (long)m.T * m.K;
    int rows[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) rows[k] = k < m.K ? perm_slot[(size_t)warp * m.K + k] : -1;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k)
        if (k < m.K && (rows[k] < 0 || rows[k] >= TK)) { bad = true; rows[k] = -1; }
    if (bad && lane == 0) set_status(status, MOE_ERR_CORRUPT_INPUT);
    for (int v = lane; v < vec_per_row; v += 32) {
        const uint4 x = u[(size_t)warp * vec_per_row + v];
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
            if (k < m.K && rows[k] >= 0) x_perm[(size_t)rows[k] * vec_per_row + v] = x;
    }
}

// One warp per permuted row: x_perm[r] = u[perm_token[r]] for the rows the offsets cover.
__global__ void gather_rows_kernel(Dims m, const uint4* __restrict__ u,
                                   const int* __restrict__ offsets,
                                   const int* __restrict__ perm_token, uint4* __restrict__ x_perm,
                                   int* status) {
    const long r = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long TK = (long)m.T * m.K;
    if (r >= TK) return;
    const int rows = offsets[m.N];
    if (r >= rows || rows > TK) return;
    const int t = perm_token[r];
    if (t < 0 || t >= m.T) {
        if (lane == 0) set_status(status, MOE_ERR_CORRUPT_INPUT);
        return;
    }
    const int vec_per_row = m.d * m.elem() / 16;
    for (int v = lane; v < vec_per_row; v += 32)
        x_perm[(size_t)r * vec_per_row + v] = u[(size_t)t * vec_per_row + v];
}

}  // namespace

cudaError_t launch_gather_rows(const Dims& m, const void* u, const int* offsets,
                               const int* perm_token, void* x_perm, int* status, cudaStream_t st) {
    const long TK = (long)m.T * m.K;
    if (TK == 0) return cudaSuccess;
    const int threads = 256;
    const long blocks = (TK * 32 + threads - 1) / threads;
    gather_rows_kernel<<<(unsigned)blocks, threads, 0, st>>>(m, static_cast<const uint4*>(u),
                                                             offsets, perm_token,
                                                             static_cast<uint4*>(x_perm), status);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_tile_hist(const Dims& m, const int* topk_idx, int* tile_counts, int* status,
                             cudaStream_t st) {
    const int n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    if (n_tiles == 0) return cudaSuccess;
    tile_hist_kernel<<<n_tiles, 256, 0, st>>>(m, topk_idx, tile_counts, status);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_perm_scan(const Dims& m, const int* tile_counts, const int* counts,
                             int* offsets, int* tile_base, int* status, cudaStream_t st) {
    const int n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    perm_scan_kernel<<<1, 256, 0, st>>>(m, n_tiles, tile_counts, counts, offsets, tile_base,
                                        status);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_perm_scatter(const Dims& m, const int* topk_idx, const int* tile_base,
                                int* perm_token, int* perm_slot, cudaStream_t st) {
    const int n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    if (n_tiles == 0) return cudaSuccess;
    const int threads = ((m.N + 31) / 32) * 32;
    perm_scatter_kernel<<<n_tiles, threads, 0, st>>>(m, topk_idx, tile_base, perm_token,
                                                     perm_slot);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gather(const Dims& m, const void* u, const int* perm_slot, void* x_perm,
                          int* status, cudaStream_t st) {
    if (m.T == 0) return cudaSuccess;
    const int threads = 256, warps_per_block = threads / 32;
    const int blocks = (m.T + warps_per_block - 1) / warps_per_block;
    gather_kernel<<<blocks, threads, 0, st>>>(m, static_cast<const uint4*>(u), perm_slot,
                                              static_cast<uint4*>(x_perm), status);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
