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
        tile_counts[(size_t)j * gridDim.x + tile] = hist[j];
}

// One CTA of 32 warps. Warp w handles experts w, w+32, ...: its lanes walk the expert's row of the
// per-tile tables ([N][n_tiles], expert-major) 32 tiles at a time, a warp scan gives each tile's
// base inside the expert (token order), and a fixed-pattern butterfly sums the tile affinity
// sums, so the result is the same on every run.
// Optional outputs: counts / psum (router totals), offsets (exclusive scan over experts), the
// balance statistics, and a check of the totals against caller-supplied counts.
__global__ void __launch_bounds__(1024) route_finalize_kernel(FinalizeArgs a) {
    __shared__ int total[kMaxRouted];
    __shared__ float ptot[kMaxRouted];
    __shared__ int off[kMaxRouted + 1];
    __shared__ float fs[kMaxRouted], Ps[kMaxRouted];
    pdl_wait();
    pdl_trigger();
    const Dims m = a.m;
    const int N = m.N, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < N; j += 32) {
        const int* cnt = a.tile_counts + (size_t)j * a.n_tiles;
        const float* ps = a.tile_psum ? a.tile_psum + (size_t)j * a.n_tiles : nullptr;
        int* tb = a.tile_base ? a.tile_base + (size_t)j * a.n_tiles : nullptr;
        int carry = 0;
        float p = 0.f;
        for (int c0 = 0; c0 < a.n_tiles; c0 += 4 * 32) {   // loads of four chunks first
            int cv[4];
            float pv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tile = c0 + q * 32 + lane;
                const bool in = tile < a.n_tiles;
                cv[q] = in ? cnt[tile] : 0;
                pv[q] = (ps && in) ? ps[tile] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tile = c0 + q * 32 + lane;
                int incl = cv[q];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (tb && tile < a.n_tiles) tb[tile] = carry + incl - cv[q];
                carry += __shfl_sync(0xffffffffu, incl, 31);
                p += pv[q];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
        if (lane == 0) {
            total[j] = carry;
            ptot[j] = p;
            if (a.counts_out) a.counts_out[j] = carry;
            if (a.psum_out) a.psum_out[j] = p;
            if (a.counts_check && a.counts_check[j] != carry)
                set_status(a.status, MOE_ERR_CORRUPT_INPUT);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && a.offsets) {
        int acc = 0;
        for (int j = 0; j < N; ++j) {
            off[j] = acc;
            acc += a.pad > 0 ? (total[j] + a.pad - 1) / a.pad * a.pad : total[j];
        }
        off[N] = acc;
    }
    __syncthreads();
    if (a.f_out || a.losses)   // f_j and P_j, then the losses from them
        for (int j = threadIdx.x; j < N; j += blockDim.x)
            balance_fp(m, total[j], ptot[j], &fs[j], &Ps[j]);
    __syncthreads();
    if (warp == 1 && a.losses) balance_losses_warp(m, fs, Ps, a.losses, lane);
    __syncthreads();
    if (a.offsets)
        for (int j = threadIdx.x; j <= N; j += blockDim.x) a.offsets[j] = off[j];
    if (a.f_out)
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            a.f_out[j] = fs[j];
            a.P_out[j] = Ps[j];
        }
}

// One CTA per 128-token tile. Each assignment a = t_local*K' + k sets bit a of its expert's
// bitmap; the row of an assignment is offsets[j] + the tile's base for j + the number of
// earlier assignments of the tile to j (a prefix popcount). Assignment order is token-major, so
// tokens stay ascending inside every expert, and the result does not depend on thread timing.
__global__ void __launch_bounds__(256) perm_scatter_kernel(Dims m, const int* __restrict__ topk_idx,
                                                         const int* __restrict__ offsets,
                                                         const int* __restrict__ tile_base,
                                                         int* __restrict__ perm_token,
                                                         int* __restrict__ perm_slot) {
    extern __shared__ uint32_t sm[];
    const int K = m.K, N = m.N, W = (kRouteTile * K + 31) / 32;   // words per expert bitmap
    uint32_t* bits = sm;                                        // [N][W]
    int* pre = reinterpret_cast<int*>(bits + (size_t)N * W);     // [N][W] popcount prefix
    int* base = pre + (size_t)N * W;                            // [N]
    const int tile = blockIdx.x, t0 = tile * kRouteTile;
    const int n = min(kRouteTile, m.T - t0) * K;
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i < N * W; i += blockDim.x) bits[i] = 0u;
    for (int j = threadIdx.x; j < N; j += blockDim.x)
        base[j] = offsets[j] + tile_base[(size_t)j * gridDim.x + tile];
    __syncthreads();
    const int* idx = topk_idx + (size_t)t0 * K;
    for (int a = threadIdx.x; a < n; a += blockDim.x) {
        const int j = idx[a];
        if (j >= 0 && j < N) atomicOr(&bits[(size_t)j * W + (a >> 5)], 1u << (a & 31));
    }
    __syncthreads();
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        int acc = 0;
        for (int w = 0; w < W; ++w) {
            pre[(size_t)j * W + w] = acc;
            acc += __popc(bits[(size_t)j * W + w]);
        }
    }
    __syncthreads();
    for (int a = threadIdx.x; a < n; a += blockDim.x) {
        const int j = idx[a];
        if (j < 0 || j >= N) {
            perm_slot[(size_t)t0 * K + a] = -1;   // flagged by the histogram
            continue;
        }
        const int w = a >> 5;
        const int rank = pre[(size_t)j * W + w] +
                         __popc(bits[(size_t)j * W + w] & ((1u << (a & 31)) - 1u));
        const int row = base[j] + rank;
        perm_token[row] = t0 + a / K;
        perm_slot[(size_t)t0 * K + a] = row;
    }
}

// One warp per token: the row is read once (16-byte vectors) and written to its K' rows.
__global__ void gather_kernel(Dims m, const uint4* __restrict__ u, const int* __restrict__ perm_slot,
                              uint4* __restrict__ x_perm, int* status, long TK) {
    pdl_wait();
    pdl_trigger();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= m.T) return;
    const int vec_per_row = m.d * m.elem() / 16;   // TK: rows of x_perm
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

// Small batches: one CTA per token, thread i copying 16-byte vectors i, i + blockDim, ... of the
// row to the token's K' rows, so the copy spreads over T SMs instead of T / 8.
__global__ void gather_cta_kernel(Dims m, const uint4* __restrict__ u,
                                  const int* __restrict__ perm_slot, uint4* __restrict__ x_perm,
                                  int* status, long TK) {
    const int t = blockIdx.x;
    const int vec_per_row = m.d * m.elem() / 16;
    // u (an input of the call, complete before its first launch) is read before the wait for
    // the predecessor's outputs, perm_slot
    uint4 x0 = make_uint4(0u, 0u, 0u, 0u);
    if ((int)threadIdx.x < vec_per_row) x0 = u[(size_t)t * vec_per_row + threadIdx.x];
    pdl_wait();
    pdl_trigger();
    int rows[kMaxTopK];
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
        rows[k] = k < m.K ? perm_slot[(size_t)t * m.K + k] : -1;
        if (k < m.K && (rows[k] < 0 || rows[k] >= TK)) {
            bad = true;
            rows[k] = -1;
        }
    }
    if (bad && threadIdx.x == 0) set_status(status, MOE_ERR_CORRUPT_INPUT);
    for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
        const uint4 x = v == (int)threadIdx.x ? x0 : u[(size_t)t * vec_per_row + v];
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
            if (k < m.K && rows[k] >= 0) x_perm[(size_t)rows[k] * vec_per_row + v] = x;
    }
}

// The rows of token t's assignments, computed by one warp. The layer call's gather places the
// assignments itself, which takes perm_scatter_kernel's work off the path that the shared
// experts' GEMM waits for. With b = t / 128, the row of (t, k) is offsets[j] + tile_base[j][b] +
// the number of assignments of the tile's earlier tokens to j = topk_idx[t][k]: a token chooses
// an expert at most once and assignments are ordered token-major, so these are the rows of
// perm_scatter_kernel's counting sort, bit for bit. rows[k] = -1 (and `bad`) for an expert id or
// a row out of range.
template <int KB>
__device__ __forceinline__ void place_token(const Dims& m, int t, const int* __restrict__ topk_idx,
                                            const int* __restrict__ offsets,
                                            const int* __restrict__ tile_base, int n_tiles,
                                            long TK, int lane, int (&rows)[KB], bool& bad) {
    const int K = m.K, N = m.N;
    const int tile = t / kRouteTile;
    int j[KB], cnt[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
        j[k] = k < K ? topk_idx[(size_t)t * K + k] : -1;
        cnt[k] = 0;
    }
    for (long a = (long)tile * kRouteTile * K + lane; a < (long)t * K; a += 32) {
        const int x = topk_idx[a];
#pragma unroll
        for (int k = 0; k < KB; ++k) cnt[k] += (x == j[k]) ? 1 : 0;
    }
    bad = false;
#pragma unroll
    for (int k = 0; k < KB; ++k) {
        const int c = __reduce_add_sync(0xffffffffu, cnt[k]);
        rows[k] = -1;
        if (k < K) {
            if (j[k] >= 0 && j[k] < N) {
                const long r = (long)offsets[j[k]] + tile_base[(size_t)j[k] * n_tiles + tile] + c;
                if (r >= 0 && r < TK) rows[k] = (int)r;
                else bad = true;
            } else {
                bad = true;
            }
        }
    }
}

// Writes the token's perm_slot entries and the perm_token entries of its rows.
template <int KB>
__device__ __forceinline__ void write_places(const Dims& m, int t, const int (&rows)[KB], int lane,
                                             int* __restrict__ perm_token,
                                             int* __restrict__ perm_slot) {
#pragma unroll
    for (int k = 0; k < KB; ++k)
        if (k < m.K && lane == k) {
            perm_slot[(size_t)t * m.K + k] = rows[k];
            if (rows[k] >= 0) perm_token[rows[k]] = t;
        }
}

// Gather with placement, one warp per token and eight tokens per CTA (a CTA's tokens lie in one
// 128-token tile). The CTA first counts, per expert, the assignments of the tile's tokens before
// its own (shared-memory histogram); warp w then adds the assignments of the CTA's tokens before
// token w to its experts, which gives the rows of place_token. The loads that do not depend on
// the histogram (the token's experts and the first rows of their segments in this tile) are issued
// before it. The token's row is then read once (16-byte vectors) and written to its K' rows.
template <int KB>
__global__ void __launch_bounds__(256) gather_place_kernel(
    Dims m, const uint4* __restrict__ u, const int* __restrict__ topk_idx,
    const int* __restrict__ offsets, const int* __restrict__ tile_base, int n_tiles,
    int* __restrict__ perm_token, int* __restrict__ perm_slot, uint4* __restrict__ x_perm,
    int* status, long TK) {
    static_assert(kRouteTile % 8 == 0, "a CTA's eight tokens lie in one tile");
    __shared__ int hist[kMaxRouted];
    pdl_wait();
    pdl_trigger();
    const int K = m.K, N = m.N;
    const int t0 = blockIdx.x * 8, lane = threadIdx.x & 31;
    const int tile = t0 / kRouteTile;
    const int t = t0 + (threadIdx.x >> 5);
    int j[KB];
    long seg0[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
        j[k] = -1;
        seg0[k] = -1;
    }
    if (t < m.T) {
#pragma unroll
        for (int k = 0; k < KB; ++k)
            if (k < K) j[k] = topk_idx[(size_t)t * K + k];
#pragma unroll
        for (int k = 0; k < KB; ++k)
            if (k < K && j[k] >= 0 && j[k] < N)
                seg0[k] = (long)offsets[j[k]] + tile_base[(size_t)j[k] * n_tiles + tile];
    }
    for (int q = threadIdx.x; q < N; q += blockDim.x) hist[q] = 0;
    __syncthreads();
    for (long a = (long)tile * kRouteTile * K + threadIdx.x; a < (long)t0 * K; a += blockDim.x) {
        const int x = topk_idx[a];
        if (x >= 0 && x < N) atomicAdd(&hist[x], 1);
    }
    __syncthreads();
    if (t >= m.T) return;
    int cnt[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) cnt[k] = 0;
    for (long a = (long)t0 * K + lane; a < (long)t * K; a += 32) {   // at most 7 K' entries
        const int x = topk_idx[a];
#pragma unroll
        for (int k = 0; k < KB; ++k) cnt[k] += (x == j[k]) ? 1 : 0;
    }
    int rows[KB];
    bool bad = false;
#pragma unroll
    for (int k = 0; k < KB; ++k) {
        const int c = __reduce_add_sync(0xffffffffu, cnt[k]);
        rows[k] = -1;
        if (k < K) {
            if (seg0[k] >= 0) {
                const long r = seg0[k] + hist[j[k]] + c;
                if (r < TK) rows[k] = (int)r;
                else bad = true;
            } else {
                bad = true;
            }
        }
    }
    if (bad && lane == 0) set_status(status, MOE_ERR_CORRUPT_INPUT);
    write_places<KB>(m, t, rows, lane, perm_token, perm_slot);
    const int vec_per_row = m.d * m.elem() / 16;
    for (int v = lane; v < vec_per_row; v += 32) {
        const uint4 x = u[(size_t)t * vec_per_row + v];
#pragma unroll
        for (int k = 0; k < KB; ++k)
            if (k < K && rows[k] >= 0) x_perm[(size_t)rows[k] * vec_per_row + v] = x;
    }
}

// The same for small batches, one CTA per token: warp 0 places the token, every thread copies.
template <int KB>
__global__ void gather_place_cta_kernel(Dims m, const uint4* __restrict__ u,
                                        const int* __restrict__ topk_idx,
                                        const int* __restrict__ offsets,
                                        const int* __restrict__ tile_base, int n_tiles,
                                        int* __restrict__ perm_token, int* __restrict__ perm_slot,
                                        uint4* __restrict__ x_perm, int* status, long TK) {
    __shared__ int rows_s[KB];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x, lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        int rows[KB];
        bool bad;
        place_token<KB>(m, t, topk_idx, offsets, tile_base, n_tiles, TK, lane, rows, bad);
        if (bad && lane == 0) set_status(status, MOE_ERR_CORRUPT_INPUT);
        write_places<KB>(m, t, rows, lane, perm_token, perm_slot);
#pragma unroll
        for (int k = 0; k < KB; ++k)
            if (lane == k) rows_s[k] = rows[k];
    }
    __syncthreads();
    int rows[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) rows[k] = k < m.K ? rows_s[k] : -1;
    const int vec_per_row = m.d * m.elem() / 16;
    for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
        const uint4 x = u[(size_t)t * vec_per_row + v];
#pragma unroll
        for (int k = 0; k < KB; ++k)
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

cudaError_t launch_route_finalize(const FinalizeArgs& a, cudaStream_t st) {
    cudaError_t e = launch_pdl(route_finalize_kernel, dim3(1), dim3(1024), 0, st, a);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_perm_scatter(const Dims& m, const int* topk_idx, const int* offsets,
                                const int* tile_base, int* perm_token, int* perm_slot,
                                cudaStream_t st) {
    const int n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    if (n_tiles == 0) return cudaSuccess;
    const int W = (kRouteTile * m.K + 31) / 32;
    const size_t smem = (size_t)m.N * W * 8 + (size_t)m.N * 4;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(perm_scatter_kernel), smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(perm_scatter_kernel, dim3(n_tiles), dim3(256), smem, st, m, topk_idx, offsets,
                   tile_base, perm_token, perm_slot);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gather(const Dims& m, const void* u, const int* perm_slot, void* x_perm,
                          int* status, cudaStream_t st, long row_limit) {
    const long rows = row_limit > 0 ? row_limit : (long)m.T * m.K;
    if (m.T == 0) return cudaSuccess;
    const int threads = 256, warps_per_block = threads / 32;
    cudaError_t e;
    if (m.T <= 2 * sm_count()) {   // a warp per token would leave most SMs idle
        const int vecs = m.d * m.elem() / 16;
        const int tpb = vecs >= 256 ? 256 : ((vecs + 31) / 32) * 32;
        e = launch_pdl(gather_cta_kernel, dim3(m.T), dim3(tpb), 0, st, m,
                       static_cast<const uint4*>(u), perm_slot, static_cast<uint4*>(x_perm), status,
                       rows);
    } else {
        const int blocks = (m.T + warps_per_block - 1) / warps_per_block;
        e = launch_pdl(gather_kernel, dim3(blocks), dim3(threads), 0, st, m,
                       static_cast<const uint4*>(u), perm_slot, static_cast<uint4*>(x_perm), status,
                       rows);
    }
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

template <int KB>
static cudaError_t launch_gather_place_kb(const Dims& m, const void* u, const int* topk_idx,
                                          const int* offsets, const int* tile_base,
                                          int* perm_token, int* perm_slot, void* x_perm,
                                          int* status, cudaStream_t st) {
    const int n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    const long TK = (long)m.T * m.K;
    if (m.T <= 2 * sm_count()) {   // a warp per token would leave most SMs idle
        const int vecs = m.d * m.elem() / 16;
        const int tpb = vecs >= 256 ? 256 : ((vecs + 31) / 32) * 32;
        return launch_pdl(gather_place_cta_kernel<KB>, dim3(m.T), dim3(tpb), 0, st, m,
                          static_cast<const uint4*>(u), topk_idx, offsets, tile_base, n_tiles,
                          perm_token, perm_slot, static_cast<uint4*>(x_perm), status, TK);
    }
    const int threads = 256, warps_per_block = threads / 32;
    const int blocks = (m.T + warps_per_block - 1) / warps_per_block;
    return launch_pdl(gather_place_kernel<KB>, dim3(blocks), dim3(threads), 0, st, m,
                      static_cast<const uint4*>(u), topk_idx, offsets, tile_base, n_tiles,
                      perm_token, perm_slot, static_cast<uint4*>(x_perm), status, TK);
}

cudaError_t launch_gather_place(const Dims& m, const void* u, const int* topk_idx,
                                const int* offsets, const int* tile_base, int* perm_token,
                                int* perm_slot, void* x_perm, int* status, cudaStream_t st) {
    if (m.T == 0) return cudaSuccess;
    cudaError_t e;
    if (m.K <= 4)
        e = launch_gather_place_kb<4>(m, u, topk_idx, offsets, tile_base, perm_token, perm_slot,
                                      x_perm, status, st);
    else if (m.K <= 8)
        e = launch_gather_place_kb<8>(m, u, topk_idx, offsets, tile_base, perm_token, perm_slot,
                                      x_perm, status, st);
    else
        e = launch_gather_place_kb<kMaxTopK>(m, u, topk_idx, offsets, tile_base, perm_token,
                                             perm_slot, x_perm, status, st);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
