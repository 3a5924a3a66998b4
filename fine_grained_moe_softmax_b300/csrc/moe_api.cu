// moe_api.cu -- the C ABI (include/moe_b300.h): argument validation, workspace layout, and the
// order of kernel launches for each entry point. No device memory is allocated here; every
// intermediate lives in the caller's workspace.
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

// Per-device side stream of the layer call and its fork / join events, created on first use (the
// first call on a device, before any graph capture of it). fork_join_mutex keeps one call's
// fork-join section from interleaving with another host thread's.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex& fork_join_mutex() {
    static std::mutex mu;
    return mu;
}

cudaError_t side_stream(SideStream** out) {
    static std::mutex mu;
    static SideStream per_dev[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    SideStream& ss = per_dev[dev];
    if (!ss.s) {
        if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess)
            return e;
    }
    *out = &ss;
    return cudaSuccess;
}

cudaError_t ensure_smem(const void* func, size_t bytes) {
    static std::mutex mu;
    static std::vector<std::pair<std::pair<const void*, int>, size_t>> granted;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (auto& g : granted)
        if (g.first.first == func && g.first.second == dev) {
            if (g.second >= bytes) return cudaSuccess;
            e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e == cudaSuccess) g.second = bytes;
            return e;
        }
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) granted.push_back({{func, dev}, bytes});
    return e;
}

// The configuration rules of every entry point (include/moe_b300.h, "Supported shapes").
int validate_config(const moe_config* c, Dims* m) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->d <= 0 || c->n_shared < 0 || c->n_routed <= 0 || c->inter <= 0 ||
        c->top_k <= 0 || c->top_k > c->n_routed || c->n_groups <= 0 ||
        c->n_groups > c->n_routed || (c->renormalize != 0 && c->renormalize != 1) ||
        (c->dtype != MOE_DTYPE_F32 && c->dtype != MOE_DTYPE_BF16) || c->skip_top < 0 ||
        c->skip_top + c->top_k > c->n_routed || (c->drop_shared != 0 && c->drop_shared != 1))
        return MOE_ERR_INVALID_ARG;
    if (c->d % 64 != 0 || c->inter % 16 != 0 || c->n_routed > kMaxRouted ||
        c->skip_top + c->top_k > kMaxTopK)
        return MOE_ERR_UNSUPPORTED;
    // row indices and element counts stay inside int32 / the tensor-map limits
    const long long TK = (long long)c->T * c->top_k;
    if (TK >= (1ll << 31) || (long long)c->n_shared * c->inter >= (1ll << 31) ||
        (long long)c->n_routed * 2 * c->inter >= (1ll << 31) ||
        (long long)c->n_routed * c->d >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED;
    m->T = c->T;
    m->d = c->d;
    m->Ks = c->n_shared;
    m->N = c->n_routed;
    m->I = c->inter;
    m->K = c->top_k;
    m->renorm = c->renormalize;
    m->D = c->n_groups;
    m->a1 = c->alpha1;
    m->a2 = c->alpha2;
    m->dtype = c->dtype;
    m->skip = c->skip_top;
    m->drop_shared = c->drop_shared;
    return MOE_OK;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_ws(const Dims& m, const void* ws, size_t ws_bytes) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MOE_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(m).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T> T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ------------------------------------------------------------------- stage timing ----

// Per recorded call: the MOE_N_STAGES + 1 stage boundaries, then the start of the gate/up launch
// over the routed groups (kEvPerCall events), and whether the shared group had a launch of its own.
constexpr int kEvPerCall = MOE_N_STAGES + 2;
struct Profile {
    std::mutex mu;
    bool on = false;
    int max_calls = 0, recorded = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<char> split;
};
Profile g_prof;

void free_profile_events() {
    for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
    g_prof.ev.clear();
    g_prof.split.clear();
    g_prof.recorded = 0;
}

// Events of the next recorded call, or null when not profiling / out of slots.
cudaEvent_t* profile_slot(char** split) {
    std::lock_guard<std::mutex> lock(g_prof.mu);
    *split = nullptr;
    if (!g_prof.on || g_prof.recorded >= g_prof.max_calls) return nullptr;
    const int c = g_prof.recorded++;
    *split = &g_prof.split[c];
    return &g_prof.ev[(size_t)c * kEvPerCall];
}

struct Marks {
    cudaEvent_t* ev;
    char* split;
    cudaStream_t st;
    void mark(int i) { mark_on(i, st); }
    void mark_on(int i, cudaStream_t s) {
        if (ev) cudaEventRecord(ev[i], s);
    }
    cudaEvent_t at(int i) { return ev ? ev[i] : nullptr; }
};

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_config* cfg) {
    Dims m;
    if (validate_config(cfg, &m) != MOE_OK) return 0;
    return ws_layout(m).total;
}

size_t moe_packed_weight_bytes(const moe_config* cfg) {
    Dims m;
    if (validate_config(cfg, &m) != MOE_OK) return 0;
    return pack_layout(m).total * (size_t)m.elem();
}

int moe_pack_weights(const moe_config* cfg, const void* w_gate, const void* w_up,
                     const void* w_down, void* packed, moe_stream_t stream) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if (!w_gate || !w_up || !w_down || !packed || !aligned16(w_gate) || !aligned16(w_up) ||
        !aligned16(w_down) || !aligned16(packed))
        return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_pack(m, w_gate, w_up, w_down, packed, (cudaStream_t)stream));
}

int moe_route(const moe_config* cfg, const void* u, const void* centroids,
              const float* logit_bias, int32_t* topk_idx, float* topk_gate, int32_t* counts,
              float* psum, void* ws, size_t ws_bytes, moe_stream_t stream) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if ((m.T > 0 && (!u || !topk_idx || !topk_gate || !aligned16(u))) || !centroids ||
        !aligned16(centroids) || !counts || !psum)
        return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(m, ws, ws_bytes)) != MOE_OK) return rc;
    const WsLayout L = ws_layout(m);
    cudaStream_t st = (cudaStream_t)stream;
    int* status = at<int>(ws, L.status);
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    cudaError_t e = launch_router(m, u, centroids, logit_bias, topk_idx, topk_gate,
                                  at<int>(ws, L.tile_counts), at<float>(ws, L.tile_psum), status,
                                  st);
    if (e == cudaSuccess) {
        FinalizeArgs fa{};
        fa.m = m;
        fa.n_tiles = L.n_tiles;
        fa.tile_counts = at<int>(ws, L.tile_counts);
        fa.tile_psum = at<float>(ws, L.tile_psum);
        fa.counts_out = counts;
        fa.psum_out = psum;
        fa.status = status;
        e = launch_route_finalize(fa, st);
    }
    return cuda_rc(e);
}

int moe_permute(const moe_config* cfg, const int32_t* topk_idx, const int32_t* counts,
                int32_t* offsets, int32_t* perm_token, int32_t* perm_slot, void* ws,
                size_t ws_bytes, moe_stream_t stream) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if ((m.T > 0 && (!topk_idx || !perm_token || !perm_slot)) || !offsets)
        return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(m, ws, ws_bytes)) != MOE_OK) return rc;
    const WsLayout L = ws_layout(m);
    cudaStream_t st = (cudaStream_t)stream;
    int* status = at<int>(ws, L.status);
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    int* tc = at<int>(ws, L.tile_counts);
    int* tb = at<int>(ws, L.tile_base);
    cudaError_t e = launch_tile_hist(m, topk_idx, tc, status, st);
    if (e == cudaSuccess) {
        FinalizeArgs fa{};
        fa.m = m;
        fa.n_tiles = L.n_tiles;
        fa.tile_counts = tc;
        fa.counts_check = counts;
        fa.offsets = offsets;
        fa.tile_base = tb;
        fa.status = status;
        e = launch_route_finalize(fa, st);
    }
    if (e == cudaSuccess)
        e = launch_perm_scatter(m, topk_idx, offsets, tb, perm_token, perm_slot, st);
    return cuda_rc(e);
}

int moe_expert_ffn(const moe_config* cfg, const void* u, const void* packed_w,
                   const int32_t* offsets, const int32_t* perm_token, void* y_routed,
                   void* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if (!packed_w || !aligned16(packed_w) || !offsets ||
        (m.T > 0 && (!u || !aligned16(u) || !perm_token || !y_routed || !aligned16(y_routed) ||
                     (m.shared_active() && (!y_shared || !aligned16(y_shared))))))
        return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(m, ws, ws_bytes)) != MOE_OK) return rc;
    const WsLayout L = ws_layout(m);
    cudaStream_t st = (cudaStream_t)stream;
    int* status = at<int>(ws, L.status);
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    cudaError_t e = launch_gather_rows(m, u, offsets, perm_token, at<void>(ws, L.x_perm), status,
                                       st);
    if (e == cudaSuccess)
        e = launch_expert_gemms(m, u, at<void>(ws, L.x_perm), packed_w, offsets,
                                at<void>(ws, L.act_r), at<void>(ws, L.act_s), y_routed, y_shared,
                                status, st, nullptr);
    return cuda_rc(e);
}

int moe_combine(const moe_config* cfg, const void* u, const void* y_routed, const void* y_shared,
                const int32_t* perm_slot, const float* topk_gate, void* h, void* ws,
                size_t ws_bytes, moe_stream_t stream) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if (m.T > 0 && (!u || !y_routed || !perm_slot || !topk_gate || !h || !aligned16(u) ||
                    !aligned16(y_routed) || !aligned16(h) || (m.shared_active() && !y_shared) ||
                    (y_shared && !aligned16(y_shared))))
        return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(m, ws, ws_bytes)) != MOE_OK) return rc;
    const WsLayout L = ws_layout(m);
    cudaStream_t st = (cudaStream_t)stream;
    int* status = at<int>(ws, L.status);
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_rc(launch_combine(m, u, y_routed, y_shared, perm_slot, topk_gate, h, status, st));
}

int moe_balance_stats(const moe_config* cfg, const int32_t* counts, const float* psum, float* f,
                      float* P, float* losses, moe_stream_t stream) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if (!counts || !psum || !f || !P || !losses) return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_balance(m, counts, psum, f, P, losses, (cudaStream_t)stream));
}

int moe_layer_forward(const moe_config* cfg, const void* u, const void* centroids,
                      const float* logit_bias, const void* packed_w, void* h, int32_t* topk_idx,
                      float* topk_gate, int32_t* counts, float* f, float* P, float* losses,
                      void* ws, size_t ws_bytes, moe_stream_t stream) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if ((m.T > 0 && (!u || !h || !topk_idx || !topk_gate || !aligned16(u) || !aligned16(h))) ||
        !centroids || !aligned16(centroids) || !packed_w || !aligned16(packed_w) || !counts ||
        !f || !P || !losses)
        return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(m, ws, ws_bytes)) != MOE_OK) return rc;
    const WsLayout L = ws_layout(m);
    cudaStream_t st = (cudaStream_t)stream;
    int* status = at<int>(ws, L.status);
    int* tc = at<int>(ws, L.tile_counts);
    float* tp = at<float>(ws, L.tile_psum);
    int* tb = at<int>(ws, L.tile_base);
    float* psum = at<float>(ws, L.psum);
    int* offsets = at<int>(ws, L.offsets);
    int* perm_token = at<int>(ws, L.perm_token);
    int* perm_slot = at<int>(ws, L.perm_slot);
    Marks mk{nullptr, nullptr, st};
    mk.ev = profile_slot(&mk.split);

    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    mk.mark(0);
    // a one-tile bf16 batch gets its routing tables from the router itself (no finalize and
    // scatter launches)
    const bool one_tile = m.dtype == MOE_DTYPE_BF16 && L.n_tiles == 1;
    SingleTileTables tab{counts, psum, offsets, perm_token, perm_slot, f, P, losses, 0};
    cudaError_t e = one_tile ? launch_router_tc(m, u, centroids, logit_bias, topk_idx, topk_gate,
                                                tc, tp, status, st, &tab)
                             : launch_router(m, u, centroids, logit_bias, topk_idx, topk_gate, tc,
                                             tp, status, st);
    mk.mark(1);
    if (e == cudaSuccess && !one_tile) {   // totals, offsets, tile bases, statistics
        FinalizeArgs fa{};
        fa.m = m;
        fa.n_tiles = L.n_tiles;
        fa.tile_counts = tc;
        fa.tile_psum = tp;
        fa.counts_out = counts;
        fa.psum_out = psum;
        fa.offsets = offsets;
        fa.tile_base = tb;
        fa.f_out = f;
        fa.P_out = P;
        fa.losses = losses;
        fa.status = status;
        e = launch_route_finalize(fa, st);
    }
    mk.mark(2);
    // With shared experts, the shared group's gate/up GEMM needs only u. The permuted token rows
    // are then placed and gathered on a side stream while it runs (the gather needs 1 KB of shared
    // memory, so its CTAs fit beside the GEMM's, and the GEMM leaves most of the memory bandwidth
    // idle); the routed groups' gate/up follows once they are ready. The gather stage of the
    // profile is then timed on the side stream and the gate/up stage is the rest of the gate/up
    // work. Several tiles: the gather also computes perm_slot / perm_token (the scatter kernel's
    // results) from the finalize kernel's offsets and tile bases; one tile: the router wrote them.
    const bool overlap = e == cudaSuccess && !one_tile && m.dtype == MOE_DTYPE_BF16 &&
                         m.shared_active();
    SideStream* ss = nullptr;
    if (overlap && (e = side_stream(&ss)) != cudaSuccess) return cuda_rc(e);
    std::unique_lock<std::mutex> fj(fork_join_mutex(), std::defer_lock);
    cudaStream_t sst = st;   // the stream of the gather
    if (overlap) {
        fj.lock();
        sst = ss->s;
        if ((e = cudaEventRecord(ss->fork, st)) == cudaSuccess)
            e = cudaStreamWaitEvent(sst, ss->fork, 0);
    }
    if (e == cudaSuccess)
        e = one_tile ? launch_gather(m, u, perm_slot, at<void>(ws, L.x_perm), status, sst)
                     : launch_gather_place(m, u, topk_idx, offsets, tb, perm_token, perm_slot,
                                           at<void>(ws, L.x_perm), status, sst);
    mk.mark_on(3, sst);
    bool joined = !overlap;
    if (overlap) {
        const cudaError_t ej = cudaEventRecord(ss->join, sst);
        if (e == cudaSuccess) e = ej;
    }
    if (mk.split) *mk.split = overlap;
    if (e == cudaSuccess) {
        joined = true;   // the routed gate/up launch waits for the join event
        e = launch_expert_gemms(m, u, at<void>(ws, L.x_perm), packed_w, offsets,
                                at<void>(ws, L.act_r), at<void>(ws, L.act_s), at<void>(ws, L.y_r),
                                at<void>(ws, L.y_s), status, st, mk.at(4),
                                overlap ? ss->join : nullptr, mk.at(MOE_N_STAGES + 1));
    }
    if (!joined) cudaStreamWaitEvent(st, ss->join, 0);   // an error: still end the fork on st
    mk.mark(5);
    if (e == cudaSuccess)
        e = launch_combine(m, u, at<void>(ws, L.y_r), at<void>(ws, L.y_s), perm_slot, topk_gate, h,
                           status, st);
    mk.mark(6);   // the statistics were produced by the finalize kernel of the permute stage
    mk.mark(7);
    return cuda_rc(e);
}

int moe_layer_routing(const moe_config* cfg, const void* ws, size_t ws_bytes,
                      const int32_t** offsets, const int32_t** perm_token,
                      const int32_t** perm_slot, const float** psum) {
    Dims m;
    int rc = validate_config(cfg, &m);
    if (rc != MOE_OK) return rc;
    if ((rc = check_ws(m, ws, ws_bytes)) != MOE_OK) return rc;
    const WsLayout L = ws_layout(m);
    void* w = const_cast<void*>(ws);
    if (offsets) *offsets = at<int>(w, L.offsets);
    if (perm_token) *perm_token = at<int>(w, L.perm_token);
    if (perm_slot) *perm_slot = at<int>(w, L.perm_slot);
    if (psum) *psum = at<float>(w, L.psum);
    return MOE_OK;
}

int moe_device_status(const void* ws, moe_stream_t stream) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    return v;
}

const char* moe_status_string(int s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_CORRUPT_INPUT: return "MOE_ERR_CORRUPT_INPUT";
        default: return "MOE_ERR_UNKNOWN";
    }
}

int moe_selftest_bounded_wait(void* ws, size_t ws_bytes, uint64_t timeout_ns,
                              moe_stream_t stream) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < 256)
        return MOE_ERR_WORKSPACE;
    const uint64_t t = timeout_ns < 1000000ull ? 1000000ull
                       : (timeout_ns > 2000000000ull ? 2000000000ull : timeout_ns);
    cudaStream_t st = (cudaStream_t)stream;
    int* status = static_cast<int*>(ws);
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_rc(launch_bounded_wait_probe(status, t, st));
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

int moe_profile_enable(int enable, int max_calls) {
    std::lock_guard<std::mutex> lock(g_prof.mu);
    free_profile_events();
    g_prof.on = false;
    if (!enable) return MOE_OK;
    if (max_calls <= 0) return MOE_ERR_INVALID_ARG;
    g_prof.ev.resize((size_t)max_calls * kEvPerCall);
    g_prof.split.assign((size_t)max_calls, 0);
    for (auto& e : g_prof.ev)
        if (cudaEventCreate(&e) != cudaSuccess) {
            e = nullptr;
            free_profile_events();
            return MOE_ERR_CUDA;
        }
    g_prof.max_calls = max_calls;
    g_prof.on = true;
    return MOE_OK;
}

int moe_profile_read(float* ms, int* n_calls) {
    if (!ms || !n_calls) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    for (int s = 0; s < MOE_N_STAGES; ++s) ms[s] = 0.f;
    for (int c = 0; c < g_prof.recorded; ++c) {
        cudaEvent_t* ev = &g_prof.ev[(size_t)c * kEvPerCall];
        if (cudaEventSynchronize(ev[MOE_N_STAGES]) != cudaSuccess) return MOE_ERR_CUDA;
        for (int s = 0; s < MOE_N_STAGES; ++s) {
            float t = 0.f;
            if (cudaEventElapsedTime(&t, ev[s], ev[s + 1]) != cudaSuccess) return MOE_ERR_CUDA;
            ms[s] += t;
        }
    }
    *n_calls = g_prof.recorded;
    return MOE_OK;
}

int moe_profile_read_gate_up(float* ms, int* n_calls, int* n_split) {
    if (!ms || !n_calls || !n_split) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    *ms = 0.f;
    *n_split = 0;
    for (int c = 0; c < g_prof.recorded; ++c) {
        cudaEvent_t* ev = &g_prof.ev[(size_t)c * kEvPerCall];
        if (cudaEventSynchronize(ev[MOE_N_STAGES]) != cudaSuccess) return MOE_ERR_CUDA;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, ev[MOE_N_STAGES + 1], ev[4]) != cudaSuccess)
            return MOE_ERR_CUDA;
        *ms += t;
        *n_split += g_prof.split[c];
    }
    *n_calls = g_prof.recorded;
    return MOE_OK;
}

}  // extern "C"
