// kernels.h -- host-side launchers of the library's kernels (internal, not part of the C ABI).
// Every launcher enqueues on `st`, returns cudaSuccess or the launch error, and bumps the launch
// counter by the number of kernels it launched.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// Checks a caller configuration against the rules every entry point applies (null, negative or
// inconsistent fields: MOE_ERR_INVALID_ARG; valid but outside this build's shapes:
// MOE_ERR_UNSUPPORTED) and fills *m on MOE_OK (moe_api.cu).
int validate_config(const moe_config* c, Dims* m);

// Router: per 128-token tile, logits, softmax, top-k, gates, tile histogram and affinity sums
// (tables expert-major: [N][n_tiles]).
cudaError_t launch_router(const Dims& m, const void* u, const void* centroids, const float* bias,
                          int* topk_idx, float* topk_gate, int* tile_counts, float* tile_psum,
                          int* status, cudaStream_t st);

// Outputs a one-tile batch (T <= 128) can get from the router directly, in place of
// launch_route_finalize + launch_perm_scatter (same values; f, P, losses may be null).
struct SingleTileTables {
    int* counts;
    float* psum;
    int* offsets;
    int* perm_token;
    int* perm_slot;
    float *f, *P, *losses;
    int pad;
};

// Tensor-core router of bf16 layers (same outputs as launch_router; with `tables`, a one-tile
// batch also gets its routing tables).
cudaError_t launch_router_tc(const Dims& m, const void* u, const void* centroids,
                             const float* bias, int* topk_idx, float* topk_gate, int* tile_counts,
                             float* tile_psum, int* status, cudaStream_t st,
                             const SingleTileTables* tables = nullptr);

// The driver's tensor-map encoder (resolved once through the runtime), or null.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// Row-major bf16 [rows, cols] as a 2D TMA map, box [box_rows x 64], 128-byte swizzle.
bool encode_bf16_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                     int box_rows);
// The same matrix as a 3D map whose box lands `chunks` consecutive [box_rows x 64] swizzled tiles
// (64-column chunks c, c+1, ...; chunk coordinate = K block index). cols % 64 == 0.
bool encode_bf16_map_chunks(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                            int box_rows, int chunks);

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
    int pad;                  // > 0: expert j's segment starts at a multiple of pad (offsets)
};
cudaError_t launch_route_finalize(const FinalizeArgs& a, cudaStream_t st);

// perm_token / perm_slot from topk_idx, the offsets and the per-tile bases.
cudaError_t launch_perm_scatter(const Dims& m, const int* topk_idx, const int* offsets,
                                const int* tile_base, int* perm_token, int* perm_slot,
                                cudaStream_t st);

// x_perm[perm_slot[t*K+k]] = u[t]; rows outside [0, row_limit) (default T*K') are corrupt.
// The layer call's gather, which also places the assignments: perm_slot / perm_token as
// perm_scatter_kernel writes them, from the finalize kernel's offsets and per-tile bases.
cudaError_t launch_gather_place(const Dims& m, const void* u, const int* topk_idx,
                                const int* offsets, const int* tile_base, int* perm_token,
                                int* perm_slot, void* x_perm, int* status, cudaStream_t st);
cudaError_t launch_gather(const Dims& m, const void* u, const int* perm_slot, void* x_perm,
                          int* status, cudaStream_t st, long row_limit = 0);

// x_perm[r] = u[perm_token[r]] for r < offsets[N].
cudaError_t launch_gather_rows(const Dims& m, const void* u, const int* offsets,
                               const int* perm_token, void* x_perm, int* status, cudaStream_t st);

// Expert GEMMs (gate/up with the SwiGLU epilogue, then down), routed groups from offsets plus one
// dense shared group. x_perm and u are the A operands of gate/up; act_r/act_s are written, then
// read by the down GEMM which writes y_r / y_s.
// With routed_ready, the shared group's gate/up runs first and the routed groups' only after
// that event (the permuted rows are produced on another stream meanwhile). Optional events:
// main_start is recorded right before the gate/up launch over the routed groups, mid_event after
// the gate/up work.
cudaError_t launch_expert_gemms(const Dims& m, const void* u, const void* x_perm,
                                const void* packed, const int* offsets, void* act_r, void* act_s,
                                void* y_r, void* y_s, int* status, cudaStream_t st,
                                cudaEvent_t mid_event, cudaEvent_t routed_ready = nullptr,
                                cudaEvent_t main_start = nullptr);

// One launch of the tensor-core grouped GEMM (bf16 in, fp32 accumulate, bf16 out): group 0 is a
// dense group of T_shared rows (when has_shared), groups 1..n_routed the routed experts (rows
// from offsets, or counts[j] rows at offsets[j] for padded segments). out = A * B^T, with
// B = rows b_rows_per_expert * j ... of b_r for routed group j. epilogue 1: the SwiGLU of the
// expert FFN (out = silu(gate) * up over the packed column pairs; pre_* receive the raw values
// when set); 2: the SwiGLU backward (the product is d_act; with the saved values pre_* of the same
// rows, out receives d_gate / d_up in packed order, row pitch ld); 0: a plain bf16 store.
struct GroupedGemm {
    const void *a_r, *a_s, *b_r, *b_s;
    uint64_t a_rows_r, a_rows_s, k_r, k_s;   // A rows and K extents
    uint64_t b_rows_r, b_rows_s;            // B total rows
    int b_rows_per_expert, n_cols_r, n_cols_s;
    void *out_r, *out_s;
    int ld_r, ld_s;
    void *pre_r, *pre_s;          // raw gate/up values (unit-major, see gemm_tc.cu)
    int pre_rows_r, pre_rows_s;   // their row counts
    int n_routed, has_shared, T_shared;
    const int* offsets;
    const int* counts;
    long max_routed_rows;
    // offsets / counts come from a launch at least two before this one, or from before the
    // call: the producer may then read them, and load the first tile's weights, before it waits
    // for the preceding launch (single-CTA tiles only)
    int preload = 0;
};
cudaError_t run_grouped_gemm(const GroupedGemm& g, int epilogue, int* status, cudaStream_t st);

// Weight-gradient GEMM C = A^T B summed over rows (see gemm_wgrad.cu). Group 0: dense over T rows
// (A_s [T, M_s], B_s [T, N_s]); routed group j: rows poff[j] .. poff[j+1]-1 of A_r [rows_r, M_r],
// B_r [rows_r, N_r] (padded, zero rows past the expert's count). mode 0 writes dW_down [E, d, I]
// (out0), mode 1 dW_gate / dW_up [E, I, d] from packed rows (out0 / out1), mode 2 dense rows
// [n_valid_rows, N_s] (out0). All fp32.
struct WgradSpec {
    const void *a_r, *b_r, *a_s, *b_s;
    uint64_t rows_r;
    int M_r, N_r, M_s, N_s;
    int n_routed, has_shared, T;
    const int* poff;
    int mode;
    float *out0, *out1;
    int Ks, I, d, n_valid_rows;
    int* tile_counter;   // device int, zero when the launch starts (dynamic tile claims)
};
cudaError_t launch_wgrad(const WgradSpec& s, int* status, cudaStream_t st);

// ---- backward helpers (backward.cu) ----
cudaError_t launch_pack_bwd(const Dims& m, const void* w_gate, const void* w_up,
                            const void* w_down, void* packed_bwd, cudaStream_t st);
cudaError_t launch_zero_pad_rows(const Dims& m, const int* poff, const int* counts, void* b0,
                                 void* b1, int width, cudaStream_t st);
cudaError_t launch_combine_bwd(const Dims& m, const void* dh, const void* y_r,
                               const int* perm_slot, const float* gate, void* d_y, float* dgate,
                               cudaStream_t st);
cudaError_t launch_du_final(const Dims& m, const void* dh, const void* dx_s, const void* du_r,
                            const void* dx, const int* perm_slot, float* du, cudaStream_t st);
cudaError_t launch_transpose_centroids(const Dims& m, int n_pad, const void* e, void* eT,
                                       cudaStream_t st);
cudaError_t launch_dbias_reduce(int N, int n_tiles, const float* tile_dz, float* d_bias,
                                cudaStream_t st);
// Router backward (router_tc.cu): recomputes the affinities of each 128-token tile and writes
// dz [T, n_pad] (bf16) = s * (ds - sum s ds), ds = gate gradient of the chosen ranks + the
// balance-loss terms (a1 f_j + a2 f'_group(j)) / T, and per-tile column sums of dz [N][n_tiles].
cudaError_t launch_router_bwd(const Dims& m, const void* u, const void* centroids,
                              const float* bias, const int* topk_idx, const float* dgate,
                              const int* counts, void* dz, float* tile_dz, int* status,
                              cudaStream_t st);

// h = u + y_s + sum_k gate * y_r[perm_slot]; rows of y_r outside [0, row_limit) (default
// T*K') are reported as corrupt and skipped.
cudaError_t launch_combine(const Dims& m, const void* u, const void* y_r, const void* y_s,
                           const int* perm_slot, const float* gate, void* h, int* status,
                           cudaStream_t st, long row_limit = 0);

// f, P, losses from counts and psum.
cudaError_t launch_balance(const Dims& m, const int* counts, const float* psum, float* f,
                          float* P, float* losses, cudaStream_t st);

// One thread waits on an mbarrier nothing arrives on; records MOE_ERR_TIMEOUT after timeout_ns.
cudaError_t launch_bounded_wait_probe(int* status, uint64_t timeout_ns, cudaStream_t st);

// Weight packing (see PackLayout).
cudaError_t launch_pack(const Dims& m, const void* w_gate, const void* w_up, const void* w_down,
                        void* packed, cudaStream_t st);

}  // namespace moe
