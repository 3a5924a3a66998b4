/*
 * moe_b300.h -- C ABI of the B300 (sm_103a) DeepSeekMoE layer-forward library.
 *
 * The layer: h_t = u_t + sum_{s < K_s} FFN_s(u_t) + sum_{k < K'} g_{t,k} FFN_{K_s + r_{t,k}}(u_t),
 * over K_s always-active shared experts and N' fine-grained routed experts, each a SwiGLU FFN of
 * intermediate width I. Routed expert r_{t,k} is the k-th best by affinity
 * s_{t,j} = softmax_j(u_t . e_j + b_j) over the N' routed experts.
 *
 * Page citations:
 *   [P1] "DeepSeekMoE 论文解读" (xxmr.cn news 118388): §两大核心策略 (fine-grained segmentation,
 *        shared-expert isolation), §方法细节：公式与负载均衡设计 (layer formula, Topk gates,
 *        expert- and device-level balance losses).
 *   [P2] "【论文总结】MoE" (mickeyding.github.io): §2.2 (centroids e_i), §2.3 (f_i, P_i, T, N',
 *        K'), §2.4 (f'_i, P'_i per device group).
 *
 * Conventions shared by every entry point:
 *   - Tensor pointers are DEVICE pointers to contiguous row-major arrays owned by the caller. The
 *     library never allocates or frees device memory; scratch lives in the caller's workspace
 *     `ws` of at least moe_workspace_bytes() bytes (256-byte aligned).
 *   - Element type of u, h, centroids and expert weights: cfg->dtype (fp32 or bf16). Gates,
 *     logit bias, affinity sums and statistics are fp32; indices and counts are int32.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     The return value reports argument and launch errors only. Errors found on the device
 *     (a bounded wait that ran out, corrupt routing input) are written to a status word inside
 *     `ws`; each call clears that word when it starts, and moe_device_status() reads it.
 *   - Supported shapes: T >= 0, d % 64 == 0, I % 16 == 0, 1 <= top_k, skip_top >= 0,
 *     skip_top + top_k <= min(N', 16), 1 <= N' <= 256, 0 <= K_s, 1 <= n_groups <= N'. Anything
 *     else returns MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED; there is no fallback path.
 *   - Calls on different streams with disjoint workspaces and outputs are independent.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,   /* null pointer, negative size, top_k > N', ... */
    MOE_ERR_UNSUPPORTED = -2,   /* valid but outside the shapes this build handles */
    MOE_ERR_WORKSPACE = -3,     /* ws_bytes < moe_workspace_bytes(cfg) or misaligned ws */
    MOE_ERR_CUDA = -4,          /* a CUDA runtime/driver call failed (launch, tensor map) */
    MOE_ERR_TIMEOUT = -5,       /* device side: a bounded wait gave up (kernel returned early) */
    MOE_ERR_CORRUPT_INPUT = -6  /* device side: routing input out of range or inconsistent */
} moe_status;

typedef enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

typedef struct {
    int32_t T;           /* tokens in this call */
    int32_t d;           /* model width */
    int32_t n_shared;    /* K_s, always-active shared experts (global ids 0..K_s-1) */
    int32_t n_routed;    /* N', routed experts (local id j, global id K_s + j) */
    int32_t inter;       /* I, intermediate width of every expert */
    int32_t top_k;       /* K', routed experts chosen per token */
    int32_t renormalize; /* 0: g = s;  1: g = s / sum over the chosen K' of s */
    int32_t n_groups;    /* D, contiguous routed-expert groups for the device-level statistic */
    float alpha1;        /* expert-level balance factor */
    float alpha2;        /* device-level balance factor */
    int32_t dtype;       /* moe_dtype of u, h, centroids and weights */
    /* Ablations of the expert-specialisation analysis ([P1] §专家特化深度分析); 0 = the layer. */
    int32_t skip_top;    /* the skip_top best-ranked routed experts of each token are disabled:
                          * the token uses ranks skip_top .. skip_top+K'-1, gates = their s */
    int32_t drop_shared; /* 1: the shared experts are disabled (no shared term in h; moe_expert_ffn
                          * leaves y_shared untouched) */
} moe_config;

/* Bytes of scratch any entry point may use for this configuration (the same figure for all). */
size_t moe_workspace_bytes(const moe_config* cfg);

/* Bytes of the packed expert-weight buffer written by moe_pack_weights. */
size_t moe_packed_weight_bytes(const moe_config* cfg);

/* Repacks caller weights into the library layout used by moe_expert_ffn / moe_layer_forward.
 *   w_gate, w_up [K_s + N', I, d]; w_down [K_s + N', d, I] (shared experts first).
 *   packed: device buffer of moe_packed_weight_bytes(cfg) bytes, written by this call.
 * One kernel launch; the caller keeps ownership of all buffers. [P1 §两大核心策略: mN experts of
 * width 1/m, K_s of them shared; the shared experts are packed as one expert of width K_s*I, which
 * computes the same sum since their gates are all 1.] */
int moe_pack_weights(const moe_config* cfg, const void* w_gate, const void* w_up,
                     const void* w_down, void* packed, moe_stream_t stream);

/* Router. For every token t: z_{t,j} = u_t . e_j + b_j (fp32 accumulation), s = softmax_j(z)
 * over the N' routed experts, the K' experts of largest s (lower index first on equal s) in rank
 * order, and their gates (s, or renormalised over the chosen K').
 *   u [T, d]; centroids [N', d]; logit_bias [N'] fp32 or NULL (treated as 0).
 *   topk_idx [T, K'] int32 routed ids in rank order; topk_gate [T, K'] fp32;
 *   counts [N'] int32: tokens that chose expert j; psum [N'] fp32: sum over t of s_{t,j}.
 * counts and psum are overwritten (not accumulated) and summed in a fixed order, so the call is
 * deterministic. [P2 §2.2: centroid affinity; P1 §方法细节: gates from Topk over s; P2 §2.3:
 * selection counts and mean affinity feed f_i and P_i] */
int moe_route(const moe_config* cfg, const void* u, const void* centroids,
              const float* logit_bias, int32_t* topk_idx, float* topk_gate, int32_t* counts,
              float* psum, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch permutation: a stable counting sort of the T*K' (token, slot) assignments by routed
 * expert, tokens ascending inside an expert.
 *   topk_idx [T, K'], counts [N'] (as produced by moe_route).
 *   offsets [N'+1]: expert j owns rows offsets[j] .. offsets[j+1]-1, offsets[N'] = T*K';
 *   perm_token [T*K']: token of each row; perm_slot [T*K']: row of assignment (t, k) at t*K'+k.
 * Expert ids outside [0, N') are skipped and counts that disagree with topk_idx are ignored in
 * favour of topk_idx; both set MOE_ERR_CORRUPT_INPUT in the status word. [Sparse activation of
 * the chosen experts, P1 §方法细节] */
int moe_permute(const moe_config* cfg, const int32_t* topk_idx, const int32_t* counts,
                int32_t* offsets, int32_t* perm_token, int32_t* perm_slot, void* ws,
                size_t ws_bytes, moe_stream_t stream);

/* Expert FFNs. Routed row r (expert j with offsets[j] <= r < offsets[j+1], token perm_token[r])
 * gets y_routed[r] = FFN_{K_s+j}(u_{perm_token[r]}); every token gets
 * y_shared[t] = sum_{s<K_s} FFN_s(u_t) (left untouched when K_s = 0).
 * FFN(x) = W_down (silu(W_gate x) * (W_up x)); bf16 inputs use tensor cores with fp32
 * accumulation and round the intermediate activation and the outputs to bf16.
 *   packed_w from moe_pack_weights; y_routed [T*K', d]; y_shared [T, d] (dtype of u).
 * [P1 §方法细节: FFN_i; P1 §两大核心策略: shared experts always active] */
int moe_expert_ffn(const moe_config* cfg, const void* u, const void* packed_w,
                   const int32_t* offsets, const int32_t* perm_token, void* y_routed,
                   void* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Gated combine with the residual, accumulated in fp32 in the fixed order u, shared, k = 0..K'-1:
 * h_t = u_t + y_shared[t] + sum_k topk_gate[t,k] * y_routed[perm_slot[t*K'+k]].
 * Rows outside [0, T*K') are skipped and set MOE_ERR_CORRUPT_INPUT.
 * [P1 §方法细节: h_t = sum_i g_{i,t} FFN_i(u_t) + u_t] */
int moe_combine(const moe_config* cfg, const void* u, const void* y_routed, const void* y_shared,
                const int32_t* perm_slot, const float* topk_gate, void* h, void* ws,
                size_t ws_bytes, moe_stream_t stream);

/* Balance statistics (fp32): f_j = N'/(K' T) counts_j, P_j = psum_j / T,
 * losses[0] = L_ExpBal = alpha1 sum_j f_j P_j,
 * losses[1] = L_DevBal = alpha2 sum_g f'_g P'_g with f'_g the mean of f and P'_g the sum of P over
 * contiguous group g (the first N' mod D groups hold one extra expert).
 *   counts [N'] int32, psum [N'] fp32 -> f [N'], P [N'], losses [2].
 * [P1 §方法细节: L_ExpBal, L_DevBal; P2 §2.3, §2.4] */
int moe_balance_stats(const moe_config* cfg, const int32_t* counts, const float* psum, float* f,
                      float* P, float* losses, moe_stream_t stream);

/* The whole layer in one call: route, permute, expert FFNs, combine and statistics.
 *   u [T, d]; centroids [N', d]; logit_bias [N'] or NULL; packed_w from moe_pack_weights;
 *   h [T, d] out; topk_idx [T, K'], topk_gate [T, K'], counts [N'], f [N'], P [N'],
 *   losses [2] out. Intermediates live in ws. [P1 §方法细节] */
int moe_layer_forward(const moe_config* cfg, const void* u, const void* centroids,
                      const float* logit_bias, const void* packed_w, void* h, int32_t* topk_idx,
                      float* topk_gate, int32_t* counts, float* f, float* P, float* losses,
                      void* ws, size_t ws_bytes, moe_stream_t stream);

/* The routing tables that the last moe_layer_forward on `ws` left in its workspace, as device
 * pointers into ws: offsets [N'+1], perm_token [T*K'] and perm_slot [T*K'] (the dispatch
 * permutation, as moe_permute returns it) and psum [N'] (sum over the call's tokens of s_{t,j},
 * as moe_route returns it; the raw sums behind P, which token-sharded callers add up across
 * ranks before moe_balance_stats). cfg must be that call's configuration (same T) and ws_bytes
 * at least moe_workspace_bytes(cfg). The pointers are valid once that call has completed on its
 * stream and until the next call that uses ws; they are read-only. Any output may be NULL.
 * Launches nothing and does not synchronise. [P2 §2.3: P_i from the affinity sums; P1 §方法细节:
 * the chosen experts' rows] */
int moe_layer_routing(const moe_config* cfg, const void* ws, size_t ws_bytes,
                      const int32_t** offsets, const int32_t** perm_token,
                      const int32_t** perm_slot, const float** psum);

/* ---- backward (training) ---- */

/* The gradients of the training objective  sum_t dh_t . h_t + L_ExpBal + L_DevBal  with respect to
 * the layer's inputs and parameters, with the expert selection and the selection counts held fixed
 * (they are piecewise constant; the balance losses act through P_j, [P1] §方法细节; [P2] §2.3-2.4).
 * bf16 layers only (fp32 configs return MOE_ERR_UNSUPPORTED). The call recomputes the forward pieces
 * it needs from u and the weights, so it needs no state from a forward call.
 *   packed_w from moe_pack_weights; packed_bwd from moe_pack_weights_backward (transposed copies
 *   of the expert weights, moe_packed_backward_bytes(cfg) bytes);
 *   dh [T, d] (layer dtype): upstream gradient of h;
 *   du [T, d] fp32; d_centroids [N', d] fp32; d_bias [N'] fp32 (gradient of the logit bias, also
 *   when logit_bias is NULL); dw_gate, dw_up [K_s+N', I, d] fp32; dw_down [K_s+N', d, I] fp32 —
 *   all overwritten; experts without tokens (or disabled ones) receive zeros.
 * ws: moe_backward_workspace_bytes(cfg) bytes, 256-byte aligned. */
size_t moe_backward_workspace_bytes(const moe_config* cfg);
size_t moe_packed_backward_bytes(const moe_config* cfg);
int moe_pack_weights_backward(const moe_config* cfg, const void* w_gate, const void* w_up,
                              const void* w_down, void* packed_bwd, moe_stream_t stream);
int moe_layer_backward(const moe_config* cfg, const void* u, const void* centroids,
                       const float* logit_bias, const void* packed_w, const void* packed_bwd,
                       const void* dh, float* du, float* d_centroids, float* d_bias,
                       float* dw_gate, float* dw_up, float* dw_down, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* A training step without the recompute: moe_layer_forward_train computes the layer forward
 * ([P1] §方法细节) with the outputs of moe_layer_forward (h, routing, f, P, losses; topk_idx,
 * topk_gate and counts may be NULL) and leaves in the backward workspace `ws` everything the
 * gradients need. moe_layer_backward_saved then computes the gradients of moe_layer_backward from
 * that state, skipping the router, permutation, gate/up and routed down GEMMs it would otherwise
 * recompute.
 *   Both calls take the same cfg (same T) and the same u, centroids and logit_bias; ws
 *   (moe_backward_workspace_bytes(cfg) bytes, 256-byte aligned) must not be used by another call
 *   in between. The backward's results equal moe_layer_backward's bit for bit; h equals
 *   moe_layer_forward's.
 *   bf16 layers only; argument and workspace errors as for moe_layer_backward. */
int moe_layer_forward_train(const moe_config* cfg, const void* u, const void* centroids,
                            const float* logit_bias, const void* packed_w, void* h,
                            int32_t* topk_idx, float* topk_gate, int32_t* counts, float* f,
                            float* P, float* losses, void* ws, size_t ws_bytes,
                            moe_stream_t stream);
int moe_layer_backward_saved(const moe_config* cfg, const void* u, const void* centroids,
                             const float* logit_bias, const void* packed_bwd, const void* dh,
                             float* du, float* d_centroids, float* d_bias, float* dw_gate,
                             float* dw_up, float* dw_down, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Waits for `stream`, then returns the device status word of `ws` (MOE_OK or a negative
 * moe_status), or MOE_ERR_CUDA if the wait itself failed. */
int moe_device_status(const void* ws, moe_stream_t stream);

/* Human-readable name of a moe_status value (static string). */
const char* moe_status_string(int status);

/* ---- permutation without a caller workspace ---- */

/* moe_permute for callers that cannot provide device scratch memory: code that runs where it may
 * not allocate (an engine that reserves all device memory up front and forbids later cudaMalloc,
 * a plugin that is handed only its input and output buffers, a latency-critical loop that cannot
 * afford the synchronisation cudaMalloc/cudaFree imply). The pages have no counterpart of this
 * call; it computes exactly what moe_permute computes, with the same arguments except `ws`.
 *   status: device int32 or NULL; cleared by the call, then set to MOE_ERR_CORRUPT_INPUT under the
 *           same conditions in which moe_permute sets its workspace status word.
 * Scratch: a fixed 1 MiB array inside this library, held on every GPU that loads the library until
 * the process exits. Limit: ceil(T / 128) * N' <= 131072 (for example T <= 65536 at N' = 256,
 * T <= 262144 at N' = 64); larger configurations return MOE_ERR_UNSUPPORTED without launching.
 * The first call on a device looks up the array's device address with that device current and
 * keeps it for the life of the process; make that first call before any stream capture, and do not
 * reset the device (cudaDeviceReset) between calls, since the address would then be stale. All
 * calls share the array: calls whose kernels can
 * overlap on a GPU (different streams, or several host threads) race and must be serialised by
 * the caller. No device memory is allocated or freed by this call. */
int moe_permute_static(const moe_config* cfg, const int32_t* topk_idx, const int32_t* counts,
                       int32_t* offsets, int32_t* perm_token, int32_t* perm_slot,
                       int32_t* status, moe_stream_t stream);

/* ---- failure detection ---- */

/* Self-test of the bounded waits that every pipelined kernel of this library uses: launches one
 * thread that waits on an mbarrier nothing ever arrives on. The wait gives up after timeout_ns
 * (clamped to [1 ms, 2 s]), writes MOE_ERR_TIMEOUT to the status word of ws and the kernel returns,
 * leaving the CUDA context usable. ws: at least 256 bytes, 256-byte aligned. Read the outcome with
 * moe_device_status(). No page describes this; it checks the library's own failure handling. */
int moe_selftest_bounded_wait(void* ws, size_t ws_bytes, uint64_t timeout_ns,
                              moe_stream_t stream);

/* ---- instrumentation (no effect on results) ---- */

/* Kernels this library has launched in this process since load (all entry points). */
uint64_t moe_launch_count(void);

/* Per-stage timing of moe_layer_forward. enable != 0 starts recording a CUDA event around each
 * stage (router, permute, gather, gate/up GEMM, down GEMM, combine, statistics) of the next
 * calls, up to max_calls of them; enable == 0 stops and frees the events. When a bf16 call with
 * shared experts and more than one router tile splits its gate/up GEMM (the shared group first,
 * beside the gather on a second stream, then the routed groups), the gather stage is its time on
 * the second stream and the gate/up stage is the time from the end of the gather to the end of
 * the routed groups' launch; the stages still add up to the call. */
int moe_profile_enable(int enable, int max_calls);

/* Waits for the recorded events and writes, per stage, the summed milliseconds over the recorded
 * calls into ms[0 .. MOE_N_STAGES-1]; *n_calls receives the number of calls recorded. */
#define MOE_N_STAGES 7
int moe_profile_read(float* ms, int* n_calls);

/* Summed milliseconds, over the recorded calls, of the gate/up GEMM launch that covers the routed
 * groups (it also covers the shared group in calls that did not split it off), from its start on
 * the call's stream to its end. *n_calls: calls recorded; *n_split: how many of them split the
 * shared group into a launch of its own. */
int moe_profile_read_gate_up(float* ms, int* n_calls, int* n_split);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
