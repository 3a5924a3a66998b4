// kernels.h -- host-side launchers of the library's kernels (internal, not part of the C ABI).
// Every launcher enqueues on `st`, returns cudaSuccess or the launch error, and bumps the launch
// counter by the number of kernels it launched.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// Router: per 128-token tile, logits, softmax, top-k, gates, tile histogram and affinity sums
// (tables expert-major: [N][n_tiles]).
cudaError_t launch_router(const Dims& m, const void* u, const void* centroids, const float* bias,
                          int* topk_idx, float* topk_gate, int* tile_counts, float* tile_psum,
                          int* status, cudaStream_t st);

// Tensor-core router of bf16 layers (same outputs as launch_router).
cudaError_t launch_router_tc(const Dims& m, const void* u, const void* centroids,
                             const float* bias, int* topk_idx, float* topk_gate, int* tile_counts,
                             float* tile_psum, int* status, cudaStream_t st);

// Row-major bf16 [rows, cols] as a 2D TMA map, box [box_rows x 64], 128-byte swizzle.
bool encode_bf16_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                     int box_rows);

// Per-tile histogram of topk_idx (used when the router's tile histogram is not at hand).
cudaError_t launch_tile_hist(const Dims& m, const int* topk_idx, int* tile_counts, int* status,
                             cudaStream_t st);

// Reduction of the per-tile router results in tile order (one CTA). Every output is optional.
struct FinalizeArgs {
    Dims m;
    int n_tiles;
    const int* tile_counts;   // [n_tiles, N]
    const float* tile_psum;   // [n_tiles, N] or null
    int* counts_out;          // [N]: tokens per expert
    float* psum_out;          // [N]: sum of affinities
    const int* counts_check;  // [N]: caller counts to verify (MOE_ERR_CORRUPT_INPUT on mismatch)
    int* offsets;             // [N+1]: exclusive scan of the totals
    int* tile_base;           // [n_tiles, N]: first row of a tile's tokens inside expert j
    float* f_out;             // [N] balance statistics
    float* P_out;             // [N]
    float* losses;            // [2]
    int* status;
};
cudaError_t launch_route_finalize(const FinalizeArgs& a, cudaStream_t st);

// perm_token / perm_slot from topk_idx, the offsets and the per-tile bases.
cudaError_t launch_perm_scatter(const Dims& m, const int* topk_idx, const int* offsets,
                                const int* tile_base, int* perm_token, int* perm_slot,
                                cudaStream_t st);

// x_perm[perm_slot[t*K+k]] = u[t].
cudaError_t launch_gather(const Dims& m, const void* u, const int* perm_slot, void* x_perm,
                          int* status, cudaStream_t st);

// x_perm[r] = u[perm_token[r]] for r < offsets[N].
cudaError_t launch_gather_rows(const Dims& m, const void* u, const int* offsets,
                               const int* perm_token, void* x_perm, int* status, cudaStream_t st);

// Expert GEMMs (gate/up with the SwiGLU epilogue, then down), routed groups from offsets plus one
// dense shared group. x_perm and u are the A operands of gate/up; act_r/act_s are written, then
// read by the down GEMM which writes y_r / y_s.
cudaError_t launch_expert_gemms(const Dims& m, const void* u, const void* x_perm,
                                const void* packed, const int* offsets, void* act_r, void* act_s,
                                void* y_r, void* y_s, int* status, cudaStream_t st,
                                cudaEvent_t mid_event);

// h = u + y_s + sum_k gate * y_r[perm_slot].
cudaError_t launch_combine(const Dims& m, const void* u, const void* y_r, const void* y_s,
                           const int* perm_slot, const float* gate, void* h, int* status,
                           cudaStream_t st);

// f, P, losses from counts and psum.
cudaError_t launch_balance(const Dims& m, const int* counts, const float* psum, float* f,
                          float* P, float* losses, cudaStream_t st);

// One thread waits on an mbarrier nothing arrives on; records MOE_ERR_TIMEOUT after timeout_ns.
cudaError_t launch_bounded_wait_probe(int* status, uint64_t timeout_ns, cudaStream_t st);

// Weight packing (see PackLayout).
cudaError_t launch_pack(const Dims& m, const void* w_gate, const void* w_up, const void* w_down,
                        void* packed, cudaStream_t st);

}  // namespace moe
