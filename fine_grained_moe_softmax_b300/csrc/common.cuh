// common.cuh -- shared device/host definitions of the MoE layer library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe_b300.h"

namespace moe {

// ---------------------------------------------------------------------------- layout ----

// Problem dimensions after validation (all int; sizes fit in int32 by the supported limits).
struct Dims {
    int T, d, Ks, N, I, K, renorm, D;
    float a1, a2;
    int dtype;        // MOE_DTYPE_F32 / MOE_DTYPE_BF16
    int skip;         // ablation: disabled top ranks per token (moe_config::skip_top)
    int drop_shared;  // ablation: shared experts disabled
    __host__ __device__ int elem() const { return dtype == MOE_DTYPE_F32 ? 4 : 2; }
    __host__ __device__ bool shared_active() const { return Ks > 0 && !drop_shared; }
};

constexpr int kRouteTile = 128;   // tokens per router / permutation tile
constexpr int kMaxRouted = 256;   // N' limit
constexpr int kMaxTopK = 16;      // K' limit

// Byte offsets of every scratch region inside the caller's workspace (256-byte aligned).
struct WsLayout {
    size_t status;        // int32 status word (+ padding)
    size_t tile_counts;   // [N, n_tiles] int32: per router tile, tokens choosing expert j
    size_t tile_psum;     // [N, n_tiles] fp32: per router tile, sum of affinities
    size_t tile_base;     // [N, n_tiles] int32: first permuted row of tile's tokens for expert j
    size_t psum;          // [N] fp32   (layer forward)
    size_t offsets;       // [N+1] int32 (layer forward)
    size_t perm_token;    // [T*K] int32 (layer forward)
    size_t perm_slot;     // [T*K] int32 (layer forward)
    size_t x_perm;        // [T*K, d] elem: token rows in permuted order
    size_t act_r;         // [T*K, I] elem: routed SwiGLU activations
    size_t act_s;         // [T, Ks*I] elem: shared SwiGLU activations
    size_t y_r;           // [T*K, d] elem (layer forward)
    size_t y_s;           // [T, d] elem (layer forward)
    size_t total;
    int n_tiles;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Routed experts rounded up to the router's MMA width (a multiple of 32).
inline int router_npad(const Dims& m) { return (m.N + 31) / 32 * 32; }

inline WsLayout ws_layout(const Dims& m) {
    WsLayout L{};
    const size_t TK = (size_t)m.T * m.K, e = (size_t)m.elem();
    L.n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    L.status = take(256);
    L.tile_counts = take((size_t)L.n_tiles * m.N * 4);
    L.tile_psum = take((size_t)L.n_tiles * m.N * 4);
    L.tile_base = take((size_t)L.n_tiles * m.N * 4);
    L.psum = take((size_t)m.N * 4);
    L.offsets = take((size_t)(m.N + 1) * 4);
    L.perm_token = take(TK * 4);
    L.perm_slot = take(TK * 4);
    L.x_perm = take(TK * m.d * e);
    L.act_r = take(TK * m.I * e);
    L.act_s = take((size_t)m.T * m.Ks * m.I * e);
    L.y_r = take(TK * m.d * e);
    L.y_s = take((size_t)m.T * m.d * e);
    L.total = o;
    return L;
}

// Packed expert weights (element offsets). Gate/up rows are interleaved in blocks of 16: packed
// row 32*b + q holds gate row 16*b + q for q < 16 and up row 16*b + q - 16 otherwise, so any
// 32-column slice of a gate/up product holds 16 gate values and their 16 matching up values.
struct PackLayout {
    size_t gu_r;   // [N, 2I, d]
    size_t gu_s;   // [2*Ks*I, d]   shared experts side by side (one expert of width Ks*I)
    size_t dn_r;   // [N, d, I]
    size_t dn_s;   // [d, Ks*I]
    size_t total;  // elements
};

inline PackLayout pack_layout(const Dims& m) {
    PackLayout P{};
    const size_t Id = (size_t)m.I * m.d;
    P.gu_r = 0;
    P.gu_s = P.gu_r + (size_t)m.N * 2 * Id;
    P.dn_r = P.gu_s + (size_t)m.Ks * 2 * Id;
    P.dn_s = P.dn_r + (size_t)m.N * Id;
    P.total = P.dn_s + (size_t)m.Ks * Id;
    return P;
}

// Transposed expert weights for the input gradients of the backward (element offsets):
//   W_down^T per routed expert [N, I, d], shared [Ks*I, d];
//   packed gate/up^T per routed expert [N, d, 2I], shared [d, 2*Ks*I] (packed column order).
struct PackBwdLayout {
    size_t wdT_r, wdT_s, wguT_r, wguT_s, total;
};

inline PackBwdLayout pack_bwd_layout(const Dims& m) {
    PackBwdLayout P{};
    const size_t Id = (size_t)m.I * m.d;
    P.wdT_r = 0;
    P.wdT_s = P.wdT_r + (size_t)m.N * Id;
    P.wguT_r = P.wdT_s + (size_t)m.Ks * Id;
    P.wguT_s = P.wguT_r + (size_t)m.N * 2 * Id;
    P.total = P.wguT_s + (size_t)m.Ks * 2 * Id;
    return P;
}

// Rows of the padded per-expert segments used by the backward: every expert's segment starts at
// a multiple of 64, so at most 63 padding rows per expert follow its T*K' real rows.
inline size_t padded_rows(const Dims& m) { return (size_t)m.T * m.K + (size_t)63 * m.N; }

// Byte offsets of the backward's scratch inside the caller's workspace (256-byte aligned).
struct BwdLayout {
    size_t status, tile_counts, tile_psum, tile_base, tile_dz;
    size_t psum, poff, counts, topk_idx, gate, perm_token, perm_slot, dgate;
    size_t x_perm, pre_r, act_r, y_r, d_y, d_gu_r, d_x_r;   // [R, .] routed rows
    size_t pre_s, act_s, d_gu_s, d_x_s, y_s;                   // [T, .] shared
    size_t dz, eT, d_u_r;
    size_t total;
    int n_tiles;
    size_t R;
};

inline BwdLayout bwd_layout(const Dims& m) {
    BwdLayout L{};
    const size_t T = m.T, K = m.K, N = m.N, d = m.d, I = m.I, KsI = (size_t)m.Ks * m.I;
    const size_t R = padded_rows(m), npad = (m.N + 31) / 32 * 32;
    L.n_tiles = (m.T + kRouteTile - 1) / kRouteTile;
    L.R = R;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    L.status = take(256);
    L.tile_counts = take((size_t)L.n_tiles * N * 4);
    L.tile_psum = take((size_t)L.n_tiles * N * 4);
    L.tile_base = take((size_t)L.n_tiles * N * 4);
    L.tile_dz = take((size_t)L.n_tiles * N * 4);
    L.psum = take(N * 4);
    L.poff = take((N + 1) * 4);
    L.counts = take(N * 4);
    L.topk_idx = take(T * K * 4);
    L.gate = take(T * K * 4);
    L.perm_token = take(R * 4);
    L.perm_slot = take(T * K * 4);
    L.dgate = take(T * K * 4);
    L.x_perm = take(R * d * 2);
    L.pre_r = take(R * 2 * I * 2);
    L.act_r = take(R * I * 2);
    L.y_r = take(R * d * 2);
    L.d_y = take(R * d * 2);
    L.d_gu_r = take(R * 2 * I * 2);
    L.d_x_r = take(R * d * 2);
    L.pre_s = take(T * 2 * KsI * 2);
    L.act_s = take(T * KsI * 2);
    L.d_gu_s = take(T * 2 * KsI * 2);
    L.d_x_s = take(T * d * 2);
    L.y_s = take(T * d * 2);   // the shared experts' output of a training forward
    L.dz = take(T * npad * 2);
    L.eT = take(d * npad * 2);
    L.d_u_r = take(T * d * 2);
    L.total = o;
    return L;
}

// ------------------------------------------------------------------------ device utils ----

// Balance statistics in one fixed order shared by every kernel that produces them:
//   f_j = N' / (K' T) count_j and P_j = psum_j / T (balance_fp, one expert at a time), then
//   L_ExpBal = a1 sum_j f_j P_j and L_DevBal = a2 sum_g mean_{j in G_g}(f_j) * sum_{j in G_g} P_j
//   over D contiguous groups, the first N' mod D one expert larger (balance_losses_warp, one whole
//   warp, from the f_j and P_j already computed).
__device__ inline void balance_fp(const Dims& m, int total_j, float ptot_j, float* f_j,
                                  float* P_j) {
    const float Tf = (float)max(m.T, 1);
    const float scale = (float)m.N / ((float)m.K * Tf);
    *f_j = scale * (float)total_j;
    *P_j = ptot_j / Tf;
}

// Called by all 32 lanes of one warp (f, P in shared memory). Lane l sums experts l, l + 32, ...
// and groups l, l + 32, ... in ascending order; a fixed butterfly adds the lanes, so every kernel
// that calls it gets the same bits. Lane 0 writes losses[0..1].
__device__ inline void balance_losses_warp(const Dims& m, const float* f, const float* P,
                                           float* losses, int lane) {
    const int N = m.N;
    float lexp = 0.f, ldev = 0.f;
    for (int j = lane; j < N; j += 32) lexp = __fmaf_rn(f[j], P[j], lexp);
    const int base = N / m.D, extra = N % m.D;
    for (int g = lane; g < m.D; g += 32) {
        const int size = base + (g < extra ? 1 : 0);
        const int first = g * base + (g < extra ? g : extra);
        float fs = 0.f, ps = 0.f;
        for (int j = first; j < first + size; ++j) {
            fs += f[j];
            ps += P[j];
        }
        ldev = __fmaf_rn(fs / (float)size, ps, ldev);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lexp += __shfl_xor_sync(0xffffffffu, lexp, o);
        ldev += __shfl_xor_sync(0xffffffffu, ldev, o);
    }
    if (lane == 0) {
        losses[0] = m.a1 * lexp;
        losses[1] = m.a2 * ldev;
    }
}

// First error wins; later errors leave the word alone.
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

template <typename E> __device__ __forceinline__ float to_f32(E x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename E> __device__ __forceinline__ E from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float silu_f32(float a) { return a / (1.0f + __expf(-a)); }

// Programmatic dependent launch. Kernels of the layer are launched so that a kernel may start
// while its predecessor in the stream finishes. pdl_wait() blocks until the predecessor grid has
// completed and its writes are visible; every kernel calls it before its first global-memory
// access (read or write) and may do only shared-memory / TMEM / barrier set-up before it.
// pdl_trigger() lets the successor be scheduled as soon as every CTA of this grid has started.
// Without a programmatic predecessor both return immediately.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------ host helpers ----

// Counts every kernel launch made through the library (moe_launch_count).
void note_launches(int n);
int sm_count();  // multiprocessors of the current device (cached per device)

// Launch with the programmatic-stream-serialization attribute (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raises the dynamic shared-memory limit of `func` on the current device to at least `bytes`;
// remembers what each (function, device) was granted so repeated launches skip the call.
cudaError_t ensure_smem(const void* func, size_t bytes);

}  // namespace moe
