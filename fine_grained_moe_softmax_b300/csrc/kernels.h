// kernels.h -- host-side launchers of the library's kernels (internal, not part of the C ABI).
// Every launcher enqueues on `st`, returns cudaSuccess or the launch error, and bumps the launch
// counter by the number of kernels it launched.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// Router: per 128-token tile, logits, softmax, top-k, gates, tile histogram and affinity sums.
cudaError_t launch_router(const Dims& m, const void* u, const void* centroids, const float* bias,
                          int* topk_idx, float* topk_gate, int* tile_counts, float* tile_psum,
                          int* status, cudaStream_t st);

// Sums the per-tile histograms and affinity sums in tile order into counts [N] and psum [N].
cudaError_t launch_route_reduce(const Dims& m, const int* tile_counts, const float* tile_psum,
                                int* counts, float* psum, cudaStream_t st);

// Per-tile histogram of topk_idx (used when the router's tile histogram is not at hand).
cudaError_t launch_tile_hist(const Dims& m, const int* topk_idx, int* tile_counts, int* status,
                             cudaStream_t st);

// Offsets [N+1] and per-tile bases from the tile histograms; checks them against `counts`
// (may be null).
cudaError_t launch_perm_scan(const Dims& m, const int* tile_counts, const int* counts,
                             int* offsets, int* tile_base, int* status, cudaStream_t st);

// perm_token / perm_slot from topk_idx and the per-tile bases.
cudaError_t launch_perm_scatter(const Dims& m, const int* topk_idx, const int* tile_base,
                                int* perm_token, int* perm_slot, cudaStream_t st);

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
