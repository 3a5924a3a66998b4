/*
 * moe_oracle.c -- CPU oracle for the DeepSeekMoE layer forward.
 *
 * TEST INFRASTRUCTURE, not part of the library. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or helper with the CUDA
 * library, and the CUDA library never calls it.
 *
 * Plain, slow, obviously correct: every value is computed in fp64 straight from its definition,
 * one token at a time. Inputs arrive as fp32 values or as bf16 bit patterns (uint16); both are
 * widened to double exactly. The only parallelism is an OpenMP loop over independent tokens; it
 * does not change the arithmetic of any token.
 *
 * Sources (pages on the DeepSeekMoE paper, ACL 2024):
 *   [P1] "DeepSeekMoE 论文解读" (xxmr.cn news 118388)
 *        §两大核心策略: fine-grained segmentation (m experts of intermediate width 1/m) and
 *                      shared-expert isolation (K_s experts always active).
 *        §方法细节：公式与负载均衡设计: h_t = sum_i g_{i,t} FFN_i(u_t) + u_t; g from
 *                      Topk({s_{j,t}}, mK); the first K_s experts are active unconditionally and
 *                      routing picks mK-K_s of the remaining mN-K_s; L_ExpBal = a1 sum f_i P_i;
 *                      L_DevBal = a2 sum over D groups of routed experts.
 *   [P2] "【论文总结】MoE" (mickeyding.github.io)
 *        §2.2: e_i is a learnable centroid per expert, scored against the token to vote top-K.
 *        §2.3: f_i = usage frequency, P_i = affinity; T tokens, N' routed experts, K' active
 *              routed experts, indicator I(.); the N'/K' factor keeps the loss independent of
 *              the expert count.
 *        §2.4: f'_i = mean usage frequency of group i's experts, P'_i = the group's affinity.
 *
 * Readings where the pages are silent or garbled (each is listed in the design notes):
 *   - residual: h = u + sum(...) (the '+' and '=' signs were lost from the printed formula);
 *   - affinity s_{t,j} = softmax over the N' routed experts of (u_t . e_j + b_j), b = optional
 *     per-expert logit bias (0 unless given);
 *   - gate g = s (default) or s / sum_topk s (renormalize = 1); shared experts have gate 1;
 *   - Top-k ranks by s descending, the lower expert index first on equal s;
 *   - FFN_i(x) = W_down,i (silu(W_gate,i x) * (W_up,i x)), silu(a) = a / (1 + exp(-a)), no biases;
 *   - f_j = N'/(K' T) count_j, P_j = (1/T) sum_t s_{t,j}; groups are contiguous routed-id ranges,
 *     the first (N' mod D) groups one expert larger; f'_g = mean of f over the group, P'_g = sum
 *     of P over the group.
 *   - ablations of "DeepSeekMoE 论文解读" §专家特化深度分析: disabling a token's top routed
 *     experts (skip_top = r) routes it to the experts ranked r+1 .. r+K' with their own affinities
 *     as gates (the softmax is unchanged); disabling the shared experts (drop_shared) removes
 *     their term from h.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

typedef struct {
    int T, d, n_shared, n_routed, inter, top_k, renormalize, n_groups;
    double alpha1, alpha2;
    int dtype;       /* ORACLE_F32: float values; ORACLE_BF16: uint16 bf16 bit patterns */
    int skip_top;    /* ablation: the skip_top best-ranked routed experts of a token are disabled */
    int drop_shared; /* ablation: 1 = the shared experts are disabled */
} oracle_cfg;

/* Exact widening of element i of an fp32 or bf16 array to double. A bf16 value is the upper
 * half of the fp32 with the same bits. */
static double elem(const void* p, int dtype, size_t i) {
    if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------- routing (one token) ---- */

/* s_{t,j} for all routed j: softmax over j of z_j = u_t . e_j + b_j.  [P2 §2.2; P1 §方法细节] */
static void token_affinity(const oracle_cfg* c, const void* u, const void* centroids,
                           const float* bias, int t, double* s) {
    const int N = c->n_routed, d = c->d;
    double zmax = -INFINITY;
    for (int j = 0; j < N; ++j) {
        double z = 0.0;
        for (int k = 0; k < d; ++k)
            z += elem(u, c->dtype, (size_t)t * d + k) * elem(centroids, c->dtype, (size_t)j * d + k);
        if (bias) z += (double)bias[j];
        s[j] = z;
        if (z > zmax) zmax = z;
    }
    double sum = 0.0;
    for (int j = 0; j < N; ++j) {
        s[j] = exp(s[j] - zmax);
        sum += s[j];
    }
    for (int j = 0; j < N; ++j) s[j] /= sum;
}

/* Order of routed experts: by affinity descending, lower index first on equal affinity. */
static void rank_experts(const double* s, int N, int* order) {
    for (int j = 0; j < N; ++j) order[j] = j;
    for (int a = 1; a < N; ++a) { /* insertion sort, stable on index */
        int x = order[a], b = a - 1;
        while (b >= 0 && s[order[b]] < s[x]) {
            order[b + 1] = order[b];
            --b;
        }
        order[b + 1] = x;
    }
}

/* Top-K' routed experts of token t in rank order, their gates, and the near-tie margin:
 * the smallest affinity gap between neighbours among ranks 1..K'+1 (ranks 1..K' if K' = N').
 * [P1 §方法细节: g_{i,t} from Topk({s_{j,t}}, mK); routing picks mK-K_s of mN-K_s experts] */
void oracle_token_route(const oracle_cfg* c, const void* u, const void* centroids,
                        const float* bias, int t, double* s, int32_t* idx, double* gate,
                        double* margin) {
    const int N = c->n_routed, K = c->top_k, r0 = c->skip_top;
    int* order = (int*)malloc(sizeof(int) * (size_t)N);
    token_affinity(c, u, centroids, bias, t, s);
    rank_experts(s, N, order);
    double topsum = 0.0;
    for (int k = 0; k < K; ++k) topsum += s[order[r0 + k]];
    for (int k = 0; k < K; ++k) {
        idx[k] = order[r0 + k];
        gate[k] = c->renormalize ? s[order[r0 + k]] / topsum : s[order[r0 + k]];
    }
    /* the chosen ranks are r0 .. r0+K-1: every neighbouring pair from rank r0-1 to r0+K decides
     * the set or its order */
    double m = INFINITY;
    const int first = r0 > 0 ? r0 - 1 : 0;
    const int last = (r0 + K < N) ? r0 + K : N - 1;
    for (int r = first; r < last; ++r) {
        double gap = s[order[r]] - s[order[r + 1]];
        if (gap < m) m = gap;
    }
    *margin = m;
    free(order);
}

/* Routing of all T tokens, then count_j = #{t : j in topk_t} and psum_j = sum_t s_{t,j}
 * (summed in token order). scores may be NULL; otherwise it receives s [T, N'].
 * [P2 §2.3: f_i counts selections via the indicator; P_i is the mean affinity] */
int oracle_route(const oracle_cfg* c, const void* u, const void* centroids, const float* bias,
                 int32_t* topk_idx, double* topk_gate, double* margin, int64_t* counts,
                 double* psum, double* scores) {
    const int T = c->T, N = c->n_routed, K = c->top_k;
    if (T < 0 || N < 1 || K < 1 || c->skip_top < 0 || c->skip_top + K > N) return -1;
    double* all_s = scores ? scores : (double*)malloc(sizeof(double) * (size_t)T * N + 1);
#pragma omp parallel for schedule(dynamic, 16)
    for (int t = 0; t < T; ++t)
        oracle_token_route(c, u, centroids, bias, t, all_s + (size_t)t * N,
                           topk_idx + (size_t)t * K, topk_gate + (size_t)t * K, margin + t);
    for (int j = 0; j < N; ++j) {
        counts[j] = 0;
        psum[j] = 0.0;
    }
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) counts[topk_idx[(size_t)t * K + k]] += 1;
        for (int j = 0; j < N; ++j) psum[j] += all_s[(size_t)t * N + j];
    }
    if (!scores) free(all_s);
    return 0;
}

/* ------------------------------------------------------------- dispatch permutation ---- */

/* Counting sort of the T*K' (token, slot) assignments by routed expert, tokens ascending inside
 * an expert. offsets [N'+1] (offsets[N'] = T*K'); perm_token[r] = token of row r;
 * perm_slot[t*K'+k] = row of assignment (t, k). Returns -1 on an out-of-range expert id. */
int oracle_permute(const oracle_cfg* c, const int32_t* topk_idx, int32_t* offsets,
                   int32_t* perm_token, int32_t* perm_slot) {
    const int T = c->T, N = c->n_routed, K = c->top_k;
    int64_t* cursor = (int64_t*)calloc((size_t)N + 1, sizeof(int64_t));
    for (size_t a = 0; a < (size_t)T * K; ++a) {
        int j = topk_idx[a];
        if (j < 0 || j >= N) {
            free(cursor);
            return -1;
        }
        cursor[j + 1] += 1;
    }
    for (int j = 0; j < N; ++j) cursor[j + 1] += cursor[j];
    for (int j = 0; j <= N; ++j) offsets[j] = (int32_t)cursor[j];
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int j = topk_idx[(size_t)t * K + k];
            int64_t r = cursor[j]++;
            perm_token[r] = t;
            perm_slot[(size_t)t * K + k] = (int32_t)r;
        }
    free(cursor);
    return 0;
}

/* --------------------------------------------------------------------- expert FFN ---- */

/* y = FFN_e(x) = W_down,e (silu(W_gate,e x) * (W_up,e x)) for global expert id e.
 * w_gate, w_up: [E, I, d]; w_down: [E, d, I].  [P1 §方法细节 FFN_i; SwiGLU reading] */
void oracle_expert_ffn(const oracle_cfg* c, const void* w_gate, const void* w_up,
                       const void* w_down, int e, const double* x, double* y) {
    const int d = c->d, I = c->inter;
    double* act = (double*)malloc(sizeof(double) * (size_t)I);
    const size_t gu0 = (size_t)e * I * d, dn0 = (size_t)e * d * I;
    for (int i = 0; i < I; ++i) {
        double a = 0.0, b = 0.0;
        for (int k = 0; k < d; ++k) {
            a += elem(w_gate, c->dtype, gu0 + (size_t)i * d + k) * x[k];
            b += elem(w_up, c->dtype, gu0 + (size_t)i * d + k) * x[k];
        }
        act[i] = a / (1.0 + exp(-a)) * b;
    }
    for (int n = 0; n < d; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += elem(w_down, c->dtype, dn0 + (size_t)n * I + i) * act[i];
        y[n] = acc;
    }
    free(act);
}

/* ----------------------------------------------------------------- layer forward ---- */

/* h for the listed tokens: h_t = u_t + sum_{s<K_s} FFN_s(u_t) + sum_k g_{t,k} FFN_{K_s+idx_k}(u_t),
 * each token routed on its own. Optional outputs: shared_out [n, d] (sum of the shared experts),
 * routed_out [n, K', d] (ungated routed expert outputs in rank order), topk_idx/topk_gate
 * [n, K'], margin [n].  [P1 §方法细节; shared isolation P1 §两大核心策略] */
int oracle_forward_tokens(const oracle_cfg* c, const void* u, const void* centroids,
                          const float* bias, const void* w_gate, const void* w_up,
                          const void* w_down, int n, const int32_t* tokens, double* h,
                          double* shared_out, double* routed_out, int32_t* topk_idx,
                          double* topk_gate, double* margin) {
    const int d = c->d, N = c->n_routed, K = c->top_k, Ks = c->n_shared;
    for (int q = 0; q < n; ++q)
        if (tokens[q] < 0 || tokens[q] >= c->T) return -1;
    if (c->skip_top < 0 || c->skip_top + K > N) return -1;
    const int n_active_shared = c->drop_shared ? 0 : Ks;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n; ++q) {
        const int t = tokens[q];
        double* x = (double*)malloc(sizeof(double) * (size_t)d);
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
        double* g = (double*)malloc(sizeof(double) * (size_t)K);
        double m;
        for (int k = 0; k < d; ++k) x[k] = elem(u, c->dtype, (size_t)t * d + k);
        oracle_token_route(c, u, centroids, bias, t, s, idx, g, &m);
        double* hq = h + (size_t)q * d;
        for (int k = 0; k < d; ++k) hq[k] = x[k];
        if (shared_out)
            for (int k = 0; k < d; ++k) shared_out[(size_t)q * d + k] = 0.0;
        for (int e = 0; e < n_active_shared; ++e) {
            oracle_expert_ffn(c, w_gate, w_up, w_down, e, x, y);
            for (int k = 0; k < d; ++k) hq[k] += y[k];
            if (shared_out)
                for (int k = 0; k < d; ++k) shared_out[(size_t)q * d + k] += y[k];
        }
        for (int r = 0; r < K; ++r) {
            oracle_expert_ffn(c, w_gate, w_up, w_down, Ks + idx[r], x, y);
            for (int k = 0; k < d; ++k) hq[k] += g[r] * y[k];
            if (routed_out)
                for (int k = 0; k < d; ++k) routed_out[((size_t)q * K + r) * d + k] = y[k];
        }
        if (topk_idx)
            for (int r = 0; r < K; ++r) topk_idx[(size_t)q * K + r] = idx[r];
        if (topk_gate)
            for (int r = 0; r < K; ++r) topk_gate[(size_t)q * K + r] = g[r];
        if (margin) margin[q] = m;
        free(x);
        free(y);
        free(s);
        free(idx);
        free(g);
    }
    return 0;
}

/* ------------------------------------------------------------- balance statistics ---- */

/* Routed experts in group g: [first, first + size), contiguous, the first (N' mod D) groups one
 * larger.  [P1 §方法细节: routed experts split into D groups, one per device] */
void oracle_group_range(int n_routed, int n_groups, int g, int* first, int* size) {
    int base = n_routed / n_groups, extra = n_routed % n_groups;
    *size = base + (g < extra ? 1 : 0);
    *first = g * base + (g < extra ? g : extra);
}

/* f_j = N'/(K'T) count_j; P_j = psum_j / T; L_ExpBal = a1 sum_j f_j P_j;
 * f'_g = mean_{j in G_g} f_j; P'_g = sum_{j in G_g} P_j; L_DevBal = a2 sum_g f'_g P'_g.
 * losses = {L_ExpBal, L_DevBal}.  [P1 §方法细节; P2 §2.3, §2.4] */
int oracle_balance_stats(const oracle_cfg* c, const int64_t* counts, const double* psum,
                         double* f, double* P, double* fg, double* Pg, double* losses) {
    const int N = c->n_routed, K = c->top_k, T = c->T, D = c->n_groups;
    if (T < 1 || D < 1 || D > N) return -1;
    double lexp = 0.0;
    for (int j = 0; j < N; ++j) {
        f[j] = (double)N / ((double)K * (double)T) * (double)counts[j];
        P[j] = psum[j] / (double)T;
        lexp += f[j] * P[j];
    }
    double ldev = 0.0;
    for (int g = 0; g < D; ++g) {
        int first, size;
        oracle_group_range(N, D, g, &first, &size);
        double fsum = 0.0, psum_g = 0.0;
        for (int j = first; j < first + size; ++j) {
            fsum += f[j];
            psum_g += P[j];
        }
        fg[g] = fsum / (double)size;
        Pg[g] = psum_g;
        ldev += fg[g] * Pg[g];
    }
    losses[0] = c->alpha1 * lexp;
    losses[1] = c->alpha2 * ldev;
    return 0;
}

/* Threads the token loops may use (1 without OpenMP). */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ backward ---- */

/* Gradients of the training objective
 *     Lambda = sum_t dh_t . h_t + L_ExpBal + L_DevBal
 * with respect to the layer inputs and parameters, for the given upstream gradient dh [T, d].
 * The expert selection and the counts (hence f_j and f'_g) are piecewise constant and are held
 * fixed, as the pages' losses use them ([P1] §方法细节: f_i is a selection frequency, P_i the
 * mean affinity; [P2] §2.3, §2.4). Per token t, with chosen experts c_k (ranks skip..skip+K'-1):
 *   h_t = u_t + sum_shared FFN_s(u_t) + sum_k g_k FFN_{c_k}(u_t)
 *   dFFN input/weights by the chain rule through y = W_d (silu(a) * b), a = W_g x, b = W_u x,
 *     silu'(a) = sig(a) (1 + a (1 - sig(a)));
 *   dgate_k = dh_t . FFN_{c_k}(u_t);  ds_j = dgate (through g = s or s / sum_chosen s)
 *            + a1 f_j / T + a2 f'_{group(j)} / T;
 *   dz_j = s_j (ds_j - sum_m s_m ds_m);  du_t += sum_j dz_j e_j;  de_j += dz_j u_t;  db_j += dz_j.
 * Outputs (all fp64, overwritten): du [T, d], d_cent [N', d], d_bias [N'], dw_gate / dw_up
 * [E, I, d], dw_down [E, d, I]. counts [N'] are the selection counts of this batch (as routed by
 * the oracle when NULL). Tokens run in order, one at a time. */
int oracle_backward(const oracle_cfg* c, const void* u, const void* centroids, const float* bias,
                    const void* w_gate, const void* w_up, const void* w_down, const double* dh,
                    const int64_t* counts_in, double* du, double* d_cent, double* d_bias,
                    double* dw_gate, double* dw_up, double* dw_down) {
    const int T = c->T, d = c->d, N = c->n_routed, K = c->top_k, I = c->inter, Ks = c->n_shared;
    const int E = Ks + N;
    if (T < 1 || c->skip_top < 0 || c->skip_top + K > N || c->n_groups < 1 || c->n_groups > N)
        return -1;
    int64_t* counts = (int64_t*)calloc((size_t)N, sizeof(int64_t));
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    double* g = (double*)malloc(sizeof(double) * (size_t)K);
    double m;
    if (counts_in) {
        for (int j = 0; j < N; ++j) counts[j] = counts_in[j];
    } else {
        for (int t = 0; t < T; ++t) {
            oracle_token_route(c, u, centroids, bias, t, s, idx, g, &m);
            for (int k = 0; k < K; ++k) counts[idx[k]] += 1;
        }
    }
    /* f_j and the group means f'_g (constants of the backward) */
    double* fj = (double*)malloc(sizeof(double) * (size_t)N);
    double* fgrp = (double*)malloc(sizeof(double) * (size_t)N);   /* f' of expert j's group */
    for (int j = 0; j < N; ++j) fj[j] = (double)N / ((double)K * (double)T) * (double)counts[j];
    for (int gi = 0; gi < c->n_groups; ++gi) {
        int first, size;
        oracle_group_range(N, c->n_groups, gi, &first, &size);
        double mean = 0.0;
        for (int j = first; j < first + size; ++j) mean += fj[j];
        mean /= (double)size;
        for (int j = first; j < first + size; ++j) fgrp[j] = mean;
    }
    memset(du, 0, sizeof(double) * (size_t)T * d);
    memset(d_cent, 0, sizeof(double) * (size_t)N * d);
    memset(d_bias, 0, sizeof(double) * (size_t)N);
    memset(dw_gate, 0, sizeof(double) * (size_t)E * I * d);
    memset(dw_up, 0, sizeof(double) * (size_t)E * I * d);
    memset(dw_down, 0, sizeof(double) * (size_t)E * d * I);

    double* x = (double*)malloc(sizeof(double) * (size_t)d);
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* b = (double*)malloc(sizeof(double) * (size_t)I);
    double* act = (double*)malloc(sizeof(double) * (size_t)I);
    double* y = (double*)malloc(sizeof(double) * (size_t)d);
    double* dy = (double*)malloc(sizeof(double) * (size_t)d);
    double* dact = (double*)malloc(sizeof(double) * (size_t)I);
    double* ds = (double*)malloc(sizeof(double) * (size_t)N);
    double* dgate = (double*)malloc(sizeof(double) * (size_t)K);

    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < d; ++k) x[k] = elem(u, c->dtype, (size_t)t * d + k);
        oracle_token_route(c, u, centroids, bias, t, s, idx, g, &m);
        const double* dht = dh + (size_t)t * d;
        double* dut = du + (size_t)t * d;
        for (int k = 0; k < d; ++k) dut[k] = dht[k];                 /* residual */
        /* experts: shared (gate 1, unless disabled) then the chosen routed ones */
        const int n_sh = c->drop_shared ? 0 : Ks;
        for (int q = 0; q < n_sh + K; ++q) {
            const int e = q < n_sh ? q : Ks + idx[q - n_sh];
            const double gate = q < n_sh ? 1.0 : g[q - n_sh];
            const size_t gu0 = (size_t)e * I * d, dn0 = (size_t)e * d * I;
            for (int i = 0; i < I; ++i) {
                double av = 0.0, bv = 0.0;
                for (int k = 0; k < d; ++k) {
                    av += elem(w_gate, c->dtype, gu0 + (size_t)i * d + k) * x[k];
                    bv += elem(w_up, c->dtype, gu0 + (size_t)i * d + k) * x[k];
                }
                a[i] = av;
                b[i] = bv;
                act[i] = av / (1.0 + exp(-av)) * bv;
            }
            if (q >= n_sh) {   /* dgate = dh . y */
                double dot = 0.0;
                for (int n = 0; n < d; ++n) {
                    double acc = 0.0;
                    for (int i = 0; i < I; ++i)
                        acc += elem(w_down, c->dtype, dn0 + (size_t)n * I + i) * act[i];
                    dot += dht[n] * acc;
                }
                dgate[q - n_sh] = dot;
            }
            for (int n = 0; n < d; ++n) dy[n] = gate * dht[n];
            for (int i = 0; i < I; ++i) {
                double acc = 0.0;
                for (int n = 0; n < d; ++n)
                    acc += elem(w_down, c->dtype, dn0 + (size_t)n * I + i) * dy[n];
                dact[i] = acc;
            }
            for (int n = 0; n < d; ++n)
                for (int i = 0; i < I; ++i) dw_down[dn0 + (size_t)n * I + i] += dy[n] * act[i];
            for (int i = 0; i < I; ++i) {
                const double sg = 1.0 / (1.0 + exp(-a[i]));
                const double silu = a[i] * sg;
                const double da = dact[i] * b[i] * sg * (1.0 + a[i] * (1.0 - sg));
                const double db = dact[i] * silu;
                for (int k = 0; k < d; ++k) {
                    dw_gate[gu0 + (size_t)i * d + k] += da * x[k];
                    dw_up[gu0 + (size_t)i * d + k] += db * x[k];
                    dut[k] += da * elem(w_gate, c->dtype, gu0 + (size_t)i * d + k) +
                              db * elem(w_up, c->dtype, gu0 + (size_t)i * d + k);
                }
            }
        }
        /* router: gates -> affinities (+ balance-loss terms) -> logits */
        for (int j = 0; j < N; ++j)
            ds[j] = (c->alpha1 * fj[j] + c->alpha2 * fgrp[j]) / (double)T;
        if (c->renormalize) {
            double S = 0.0, w = 0.0;
            for (int k = 0; k < K; ++k) S += s[idx[k]];
            for (int k = 0; k < K; ++k) w += dgate[k] * s[idx[k]];
            for (int k = 0; k < K; ++k) ds[idx[k]] += dgate[k] / S - w / (S * S);
        } else {
            for (int k = 0; k < K; ++k) ds[idx[k]] += dgate[k];
        }
        double sds = 0.0;
        for (int j = 0; j < N; ++j) sds += s[j] * ds[j];
        for (int j = 0; j < N; ++j) {
            const double dz = s[j] * (ds[j] - sds);
            d_bias[j] += dz;
            for (int k = 0; k < d; ++k) {
                dut[k] += dz * elem(centroids, c->dtype, (size_t)j * d + k);
                d_cent[(size_t)j * d + k] += dz * x[k];
            }
        }
    }
    free(counts); free(s); free(idx); free(g); free(fj); free(fgrp); free(x); free(a); free(b);
    free(act); free(y); free(dy); free(dact); free(ds); free(dgate);
    return 0;
}
