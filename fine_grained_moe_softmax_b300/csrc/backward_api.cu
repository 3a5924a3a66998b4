// backward_api.cu -- C ABI of the layer backward and of the training pair (include/moe_b300.h):
// argument checks and the order of launches. The stateless backward recomputes the forward pieces
// it needs from the inputs, then runs the chain rule stage by stage. The training forward
// computes those pieces once, together with the layer output, and the saved backward starts from
// them. All intermediates live in the caller's workspace.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

int check_bwd(const moe_config* c, Dims* m) {
    const int rc = validate_config(c, m);
    if (rc != MOE_OK) return rc;
    return c->dtype == MOE_DTYPE_BF16 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename T> T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace moe {
namespace {

// mode 0: recompute the forward state, then the gradients (moe_layer_backward); mode 1: the
// forward state plus the shared experts' outputs, the combine and the balance statistics, leaving
// the state in ws (moe_layer_forward_train); mode 2: the gradients from the state a mode-1 call
// left in ws (moe_layer_backward_saved).
int layer_train(int mode, const moe_config* cfg, const void* u, const void* centroids,
                const float* logit_bias, const void* packed_w, const void* packed_bwd,
                const void* dh, void* h, int32_t* topk_idx_out, float* topk_gate_out,
                int32_t* counts_out, float* f, float* P, float* losses, float* du,
                float* d_centroids, float* d_bias, float* dw_gate, float* dw_up, float* dw_down,
                void* ws, size_t ws_bytes, cudaStream_t st) {
    Dims m;
    int rc = check_bwd(cfg, &m);
    if (rc != MOE_OK) return rc;
    const bool fwd = mode != 2, grads = mode != 1;
    if (!centroids || !a16(centroids) || (m.T > 0 && (!u || !a16(u))))
        return MOE_ERR_INVALID_ARG;
    if (fwd && (!packed_w || !a16(packed_w))) return MOE_ERR_INVALID_ARG;
    if (mode == 1 && ((m.T > 0 && (!h || !a16(h))) || !f || !P || !losses))
        return MOE_ERR_INVALID_ARG;
    if (grads && (!packed_bwd || !a16(packed_bwd) || !d_centroids || !d_bias || !dw_gate ||
                  !dw_up || !dw_down || !a16(dw_gate) || !a16(dw_up) || !a16(dw_down) ||
                  !a16(d_centroids) || (m.T > 0 && (!dh || !a16(dh) || !du || !a16(du)))))
        return MOE_ERR_INVALID_ARG;
    const BwdLayout L = bwd_layout(m);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < L.total)
        return MOE_ERR_WORKSPACE;
    const size_t E = (size_t)m.Ks + m.N, Id = (size_t)m.I * m.d;
    int* status = at<int>(ws, L.status);
    // the status word and the tile counters of the three weight-gradient launches
    if (cudaMemsetAsync(status, 0, 4 * sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (mode == 1 && m.T == 0) {   // no token: zero statistics, nothing else to produce
        if (cudaMemsetAsync(f, 0, (size_t)m.N * 4, st) != cudaSuccess ||
            cudaMemsetAsync(P, 0, (size_t)m.N * 4, st) != cudaSuccess ||
            cudaMemsetAsync(losses, 0, 2 * 4, st) != cudaSuccess ||
            (counts_out && cudaMemsetAsync(counts_out, 0, (size_t)m.N * 4, st) != cudaSuccess))
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (grads && (m.T == 0 || !m.shared_active())) {
        // no token gives a gradient to the disabled (or any, when T = 0) experts
        const size_t n_zero = m.T == 0 ? E : (size_t)m.Ks;
        if (cudaMemsetAsync(dw_gate, 0, n_zero * Id * 4, st) != cudaSuccess ||
            cudaMemsetAsync(dw_up, 0, n_zero * Id * 4, st) != cudaSuccess ||
            cudaMemsetAsync(dw_down, 0, n_zero * Id * 4, st) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    if (m.T == 0) {
        if (cudaMemsetAsync(d_centroids, 0, (size_t)m.N * m.d * 4, st) != cudaSuccess ||
            cudaMemsetAsync(d_bias, 0, (size_t)m.N * 4, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const PackLayout PL = pack_layout(m);
    const PackBwdLayout Q = pack_bwd_layout(m);
    const char* pw = static_cast<const char*>(packed_w);
    const char* pb = static_cast<const char*>(packed_bwd);
    const uint64_t R = L.R, T = m.T, I = m.I, d = m.d, KsI = (uint64_t)m.Ks * m.I;
    const int n_pad = router_npad(m);
    const bool shared = m.shared_active();
    int* poff = at<int>(ws, L.poff);
    int* counts = at<int>(ws, L.counts);
    int* topk_idx = at<int>(ws, L.topk_idx);
    float* gate = at<float>(ws, L.gate);
    int* perm_slot = at<int>(ws, L.perm_slot);
    void* x_perm = at<void>(ws, L.x_perm);
    void* act_r = at<void>(ws, L.act_r);
    void* act_s = at<void>(ws, L.act_s);
    void* d_y = at<void>(ws, L.d_y);
    void* d_gu_r = at<void>(ws, L.d_gu_r);
    void* d_gu_s = at<void>(ws, L.d_gu_s);

    GroupedGemm g{};
    g.n_routed = m.N;
    g.has_shared = shared;
    g.T_shared = m.T;
    g.offsets = poff;
    g.counts = counts;
    g.max_routed_rows = (long)R;

    // ---- forward state, routed rows in padded per-expert segments ----
    cudaError_t e = cudaSuccess;
    if (fwd)
        e = launch_router(m, u, centroids, logit_bias, topk_idx, gate, at<int>(ws, L.tile_counts),
                          at<float>(ws, L.tile_psum), status, st);
    if (fwd && e == cudaSuccess) {
        FinalizeArgs fa{};
        fa.m = m;
        fa.n_tiles = L.n_tiles;
        fa.tile_counts = at<int>(ws, L.tile_counts);
        fa.tile_psum = at<float>(ws, L.tile_psum);
        fa.counts_out = counts;
        fa.psum_out = at<float>(ws, L.psum);
        fa.offsets = poff;
        fa.tile_base = at<int>(ws, L.tile_base);
        fa.status = status;
        fa.pad = 64;
        if (mode == 1) {   // the balance statistics of this batch
            fa.f_out = f;
            fa.P_out = P;
            fa.losses = losses;
        }
        e = launch_route_finalize(fa, st);
    }
    if (fwd && e == cudaSuccess)
        e = launch_perm_scatter(m, topk_idx, poff, at<int>(ws, L.tile_base),
                                at<int>(ws, L.perm_token), perm_slot, st);
    if (fwd && e == cudaSuccess) e = launch_gather(m, u, perm_slot, x_perm, status, st, (long)R);
    if (fwd && e == cudaSuccess)
        e = launch_zero_pad_rows(m, poff, counts, x_perm, d_y, (int)d, st);
    if (fwd && e == cudaSuccess)
        e = launch_zero_pad_rows(m, poff, counts, act_r, nullptr, (int)I, st);
    if (fwd && e == cudaSuccess) {   // gate/up with the SwiGLU epilogue, keeping the raw values
        GroupedGemm gu = g;
        gu.a_r = x_perm;
        gu.a_s = u;
        gu.b_r = pw + PL.gu_r * 2;
        gu.b_s = pw + PL.gu_s * 2;
        gu.a_rows_r = R;
        gu.a_rows_s = T;
        gu.k_r = gu.k_s = d;
        gu.b_rows_r = (uint64_t)m.N * 2 * I;
        gu.b_rows_s = 2 * KsI;
        gu.b_rows_per_expert = (int)(2 * I);
        gu.n_cols_r = (int)(2 * I);
        gu.n_cols_s = (int)(2 * KsI);
        gu.out_r = act_r;
        gu.out_s = act_s;
        gu.ld_r = (int)I;
        gu.ld_s = (int)KsI;
        gu.pre_r = at<void>(ws, L.pre_r);
        gu.pre_s = at<void>(ws, L.pre_s);
        gu.pre_rows_r = (int)R;
        gu.pre_rows_s = (int)T;
        e = run_grouped_gemm(gu, 1, status, st);
    }
    if (fwd && e == cudaSuccess) {   // routed expert outputs (also for the gate gradients)
        GroupedGemm dn = g;
        dn.has_shared = mode == 1 && shared;   // the shared experts only for the layer output
        dn.a_r = act_r;
        dn.a_s = act_s;
        dn.b_r = pw + PL.dn_r * 2;
        dn.b_s = pw + PL.dn_s * 2;
        dn.a_rows_r = R;
        dn.a_rows_s = T;
        dn.k_r = I;
        dn.k_s = KsI;
        dn.b_rows_r = (uint64_t)m.N * d;
        dn.b_rows_s = d;
        dn.b_rows_per_expert = (int)d;
        dn.n_cols_r = dn.n_cols_s = (int)d;
        dn.out_r = at<void>(ws, L.y_r);
        dn.out_s = at<void>(ws, L.y_s);
        dn.ld_r = dn.ld_s = (int)d;
        e = run_grouped_gemm(dn, 0, status, st);
    }
    if (mode == 1) {   // h = u + shared outputs + gated routed outputs, and the routing outputs
        if (e == cudaSuccess)
            e = launch_combine(m, u, at<void>(ws, L.y_r), at<void>(ws, L.y_s), perm_slot, gate, h,
                               status, st, (long)R);
        const size_t tk = (size_t)m.T * m.K;
        if (e == cudaSuccess && topk_idx_out)
            e = cudaMemcpyAsync(topk_idx_out, topk_idx, tk * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && topk_gate_out)
            e = cudaMemcpyAsync(topk_gate_out, gate, tk * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && counts_out)
            e = cudaMemcpyAsync(counts_out, counts, (size_t)m.N * 4, cudaMemcpyDeviceToDevice,
                                st);
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }

    // ---- backward ----
    if (e == cudaSuccess)
        e = launch_combine_bwd(m, dh, at<void>(ws, L.y_r), perm_slot, gate, d_y,
                               at<float>(ws, L.dgate), st);
    if (e == cudaSuccess)
        e = launch_router_bwd(m, u, centroids, logit_bias, topk_idx, at<float>(ws, L.dgate),
                              counts, at<void>(ws, L.dz), at<float>(ws, L.tile_dz), status, st);
    if (e == cudaSuccess)
        e = launch_dbias_reduce(m.N, L.n_tiles, at<float>(ws, L.tile_dz), d_bias, st);
    if (e == cudaSuccess) e = launch_transpose_centroids(m, n_pad, centroids, at<void>(ws, L.eT), st);
    if (e == cudaSuccess) {   // router part of du: dz [T, n_pad] x e
        GroupedGemm gr{};
        gr.n_routed = 0;
        gr.has_shared = 1;
        gr.T_shared = m.T;
        gr.a_s = at<void>(ws, L.dz);
        gr.b_s = at<void>(ws, L.eT);
        gr.a_rows_s = T;
        gr.k_s = (uint64_t)n_pad;
        gr.b_rows_s = d;
        gr.n_cols_s = (int)d;
        gr.out_s = at<void>(ws, L.d_u_r);
        gr.ld_s = (int)d;
        e = run_grouped_gemm(gr, 0, status, st);
    }
    if (e == cudaSuccess) {   // centroid gradient: dz^T u
        WgradSpec w{};
        w.a_s = at<void>(ws, L.dz);
        w.b_s = u;
        w.M_s = n_pad;
        w.N_s = (int)d;
        w.has_shared = 1;
        w.n_routed = 0;
        w.T = m.T;
        w.mode = 2;
        w.tile_counter = status + 1;
        w.out0 = d_centroids;
        w.n_valid_rows = m.N;
        e = launch_wgrad(w, status, st);
    }
    if (e == cudaSuccess) {   // d_act = d_y W_down (routed), dh W_down (shared), then the
                              // SwiGLU backward in the epilogue: d_gu (packed gate/up order)
        GroupedGemm dd = g;
        dd.a_r = d_y;
        dd.a_s = dh;
        dd.b_r = pb + Q.wdT_r * 2;
        dd.b_s = pb + Q.wdT_s * 2;
        dd.a_rows_r = R;
        dd.a_rows_s = T;
        dd.k_r = dd.k_s = d;
        dd.b_rows_r = (uint64_t)m.N * I;
        dd.b_rows_s = KsI;
        dd.b_rows_per_expert = (int)I;
        dd.n_cols_r = (int)I;
        dd.n_cols_s = (int)KsI;
        dd.out_r = d_gu_r;
        dd.out_s = d_gu_s;
        dd.ld_r = (int)(2 * I);
        dd.ld_s = (int)(2 * KsI);
        dd.pre_r = at<void>(ws, L.pre_r);
        dd.pre_s = at<void>(ws, L.pre_s);
        dd.pre_rows_r = (int)R;
        dd.pre_rows_s = (int)T;
        e = run_grouped_gemm(dd, 2, status, st);
    }
    if (e == cudaSuccess)   // rows past each expert's count carry no gradient
        e = launch_zero_pad_rows(m, poff, counts, d_gu_r, nullptr, (int)(2 * I), st);
    if (e == cudaSuccess) {   // d_x = d_gu [W_gate; W_up] (packed order)
        GroupedGemm dx = g;
        dx.a_r = d_gu_r;
        dx.a_s = d_gu_s;
        dx.b_r = pb + Q.wguT_r * 2;
        dx.b_s = pb + Q.wguT_s * 2;
        dx.a_rows_r = R;
        dx.a_rows_s = T;
        dx.k_r = 2 * I;
        dx.k_s = 2 * KsI;
        dx.b_rows_r = (uint64_t)m.N * d;
        dx.b_rows_s = d;
        dx.b_rows_per_expert = (int)d;
        dx.n_cols_r = dx.n_cols_s = (int)d;
        dx.out_r = at<void>(ws, L.d_x_r);
        dx.out_s = at<void>(ws, L.d_x_s);
        dx.ld_r = dx.ld_s = (int)d;
        e = run_grouped_gemm(dx, 0, status, st);
    }
    if (e == cudaSuccess) {   // dW_down = d_y^T act per expert (shared: dh^T act_s)
        WgradSpec w{};
        w.a_r = d_y;
        w.b_r = act_r;
        w.rows_r = R;
        w.M_r = (int)d;
        w.N_r = (int)I;
        w.a_s = dh;
        w.b_s = act_s;
        w.M_s = (int)d;
        w.N_s = (int)KsI;
        w.n_routed = m.N;
        w.has_shared = shared;
        w.T = m.T;
        w.poff = poff;
        w.mode = 0;
        w.tile_counter = status + 2;
        w.out0 = dw_down;
        w.Ks = m.Ks;
        w.I = m.I;
        w.d = m.d;
        e = launch_wgrad(w, status, st);
    }
    if (e == cudaSuccess) {   // dW_gate, dW_up = d_gu^T x per expert (shared: d_gu_s^T u)
        WgradSpec w{};
        w.a_r = d_gu_r;
        w.b_r = x_perm;
        w.rows_r = R;
        w.M_r = (int)(2 * I);
        w.N_r = (int)d;
        w.a_s = d_gu_s;
        w.b_s = u;
        w.M_s = (int)(2 * KsI);
        w.N_s = (int)d;
        w.n_routed = m.N;
        w.has_shared = shared;
        w.T = m.T;
        w.poff = poff;
        w.mode = 1;
        w.tile_counter = status + 3;
        w.out0 = dw_gate;
        w.out1 = dw_up;
        w.Ks = m.Ks;
        w.I = m.I;
        w.d = m.d;
        e = launch_wgrad(w, status, st);
    }
    if (e == cudaSuccess)
        e = launch_du_final(m, dh, at<void>(ws, L.d_x_s), at<void>(ws, L.d_u_r),
                            at<void>(ws, L.d_x_r), perm_slot, du, st);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_backward_workspace_bytes(const moe_config* cfg) {
    Dims m;
    if (check_bwd(cfg, &m) != MOE_OK) return 0;
    return bwd_layout(m).total;
}

size_t moe_packed_backward_bytes(const moe_config* cfg) {
    Dims m;
    if (check_bwd(cfg, &m) != MOE_OK) return 0;
    return pack_bwd_layout(m).total * 2;
}

int moe_pack_weights_backward(const moe_config* cfg, const void* w_gate, const void* w_up,
                              const void* w_down, void* packed_bwd, moe_stream_t stream) {
    Dims m;
    int rc = check_bwd(cfg, &m);
    if (rc != MOE_OK) return rc;
    if (!w_gate || !w_up || !w_down || !packed_bwd || !a16(packed_bwd)) return MOE_ERR_INVALID_ARG;
    return launch_pack_bwd(m, w_gate, w_up, w_down, packed_bwd, (cudaStream_t)stream) ==
                   cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_layer_backward(const moe_config* cfg, const void* u, const void* centroids,
                       const float* logit_bias, const void* packed_w, const void* packed_bwd,
                       const void* dh, float* du, float* d_centroids, float* d_bias,
                       float* dw_gate, float* dw_up, float* dw_down, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
    return layer_train(0, cfg, u, centroids, logit_bias, packed_w, packed_bwd, dh, nullptr,
                       nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, du, d_centroids,
                       d_bias, dw_gate, dw_up, dw_down, ws, ws_bytes, (cudaStream_t)stream);
}

int moe_layer_forward_train(const moe_config* cfg, const void* u, const void* centroids,
                            const float* logit_bias, const void* packed_w, void* h,
                            int32_t* topk_idx, float* topk_gate, int32_t* counts, float* f,
                            float* P, float* losses, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
    return layer_train(1, cfg, u, centroids, logit_bias, packed_w, nullptr, nullptr, h, topk_idx,
                       topk_gate, counts, f, P, losses, nullptr, nullptr, nullptr, nullptr,
                       nullptr, nullptr, ws, ws_bytes, (cudaStream_t)stream);
}

int moe_layer_backward_saved(const moe_config* cfg, const void* u, const void* centroids,
                             const float* logit_bias, const void* packed_bwd, const void* dh,
                             float* du, float* d_centroids, float* d_bias, float* dw_gate,
                             float* dw_up, float* dw_down, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
    return layer_train(2, cfg, u, centroids, logit_bias, nullptr, packed_bwd, dh, nullptr,
                       nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, du, d_centroids,
                       d_bias, dw_gate, dw_up, dw_down, ws, ws_bytes, (cudaStream_t)stream);
}

}  // extern "C"
