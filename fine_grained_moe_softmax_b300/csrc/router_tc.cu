// router_tc.cu -- router of bf16 layers on the tensor cores.
//
// [P1] "DeepSeekMoE 论文解读" (xxmr.cn), §方法细节: gates come from Topk({s_{j,t}}, mK) over the
//      routed experts (the K_s shared experts are always active and are not ranked).
// [P2] "【论文总结】MoE" (mickeyding.github.io), §2.2: s_{j,t} = softmax_j(u_t . e_j) against the
//      learnable centroids e_j; §2.3: f_i counts selections, P_i averages s over the T tokens.
//
// The logits of a 128-token tile are one [128 x d] x [d x N'] product: the tile's token rows and
// the centroids stream through a TMA ring into tcgen05.mma (M = 128, N = N' rounded up to 32),
// accumulating fp32 logits in TMEM. When there are few tiles (decode-sized batches), a cluster of
// C CTAs shares a tile, each over 1/C of d; the other CTAs leave their partial logits in their
// shared memory and the first adds them to its own, in rank order, through distributed shared
// memory, so the sum does not depend on timing. Four epilogue warps then own one token per thread: each reads
// its logit row from TMEM once (warp w sees TMEM lanes 32*(w%4) .. +31), adds the optional bias,
// keeps the row in the (by then idle) TMA ring, and computes the softmax, a register top-K'
// (ranked by logit; the lower index wins ties), the gates, the tile's expert histogram and, by a
// warp transpose-reduction, the tile's per-expert sums of affinities in a fixed order.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "waits.cuh"

namespace moe {

namespace {

constexpr int RBM = 128;
constexpr int RBK = 64;
constexpr int kThreads = 192;
constexpr int kMaxStages = 8;

struct RouterArgs {
    CUtensorMap a;        // u [T, d], box [128 x 64]
    CUtensorMap b;        // centroids [N', d], box [n_pad x 64]
    const float* bias;    // [N'] or null
    int T, N, K, renorm, skip, k_blocks, n_pad, stages, tmem_cols;
    int csize;            // CTAs per tile (cluster size); CTA r takes K blocks [r kb/C, (r+1) kb/C)
    uint32_t stage_bytes;
    int* topk_idx;
    float* topk_gate;
    int* tile_counts;
    float* tile_psum;
    int* status;
    // backward mode
    const float* dgate;   // [T, K'] gradient of the chosen gates
    const int* counts;    // [N'] selection counts of the batch (f_j)
    __nv_bfloat16* dz;    // [T, n_pad] out
    float* tile_dz;       // [N'][n_tiles] out: per-tile sums of dz
    float a1, a2;
    int D;
    // a batch of one tile (T <= 128) can finish its routing tables here, in place of the finalize
    // and scatter kernels: fused != 0 and the outputs below
    int fused, pad;
    Dims dims;
    int* counts_out;      // [N']
    float* psum_out;      // [N']
    int* offsets;         // [N' + 1]
    int* perm_token;      // [T K']
    int* perm_slot;       // [T K']
    float *f_out, *P_out, *losses;   // balance statistics, or null
};

template <int KMAX>
struct TopK {
    float v[KMAX];
    int i[KMAX];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int q = 0; q < KMAX; ++q) {
            v[q] = -INFINITY;
            i[q] = -1;
        }
    }
    // candidates arrive in ascending expert index; only a strictly larger value displaces
    __device__ __forceinline__ void push(float x, int j) {
        if (!(x > v[KMAX - 1])) return;
#pragma unroll
        for (int q = KMAX - 1; q > 0; --q) {
            if (x > v[q]) {
                if (x > v[q - 1]) {
                    v[q] = v[q - 1];
                    i[q] = i[q - 1];
                } else {
                    v[q] = x;
                    i[q] = j;
                }
            }
        }
        if (x > v[0]) {
            v[0] = x;
            i[0] = j;
        }
    }
};

// One halving step of the warp transpose-reduction: lanes with bit HALF clear keep columns
// [0, HALF) of their block and receive the partner's; lanes with it set keep [HALF, 2*HALF).
template <int HALF>
__device__ __forceinline__ void halve(float (&v)[32], bool upper) {
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
        const float send = upper ? v[i] : v[i + HALF];
        const float keep = upper ? v[i + HALF] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, HALF);
    }
}

// After this, lane l of the warp holds the sum over the 32 lanes of column l of v[0..31].
__device__ __forceinline__ float column_sums(float (&v)[32], int lane) {
    halve<16>(v, lane & 16);
    halve<8>(v, lane & 8);
    halve<4>(v, lane & 4);
    halve<2>(v, lane & 2);
    halve<1>(v, lane & 1);
    return v[0];
}

__device__ __forceinline__ void epilogue_bar() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// The routing tables of a one-tile batch, by the four epilogue warps (et = 0..127, thread et = token
// et) after the tile is routed: totals, offsets (exclusive scan, segments padded to a.pad), the
// balance statistics and the stable permutation. The rank of token t in expert j is the number of
// earlier tokens of the tile choosing j (a prefix popcount of j's token bitmap); these are the
// results of the finalize and scatter kernels for the same batch, bit for bit. `scratch` is the
// idle TMA ring. Every epilogue warp runs the whole sequence (the barriers need all four).
__device__ __noinline__ void finish_single_tile(const RouterArgs& a, uint8_t* scratch,
                                                const int* hist, const float* colsum,
                                                const int* chosen, int et, int lane) {
    const int N = a.N, K = a.K, T = a.T;
    uint32_t* bits = reinterpret_cast<uint32_t*>(scratch);         // [N'][4]: tokens 0..127
    int* off = reinterpret_cast<int*>(bits + 4 * kMaxRouted);       // [N' + 1]
    float* ptot = reinterpret_cast<float*>(off + kMaxRouted + 1);   // [N']
    float* fs = ptot + kMaxRouted;                                  // [N']
    float* Ps = fs + kMaxRouted;                                    // [N']
    for (int i = et; i < 4 * N; i += 128) bits[i] = 0u;
    for (int j = et; j < N; j += 128) {
        const float col = ((colsum[j] + colsum[kMaxRouted + j]) + colsum[2 * kMaxRouted + j]) +
                          colsum[3 * kMaxRouted + j];
        ptot[j] = col;
        a.counts_out[j] = hist[j];
        a.psum_out[j] = col;
        balance_fp(a.dims, hist[j], col, &fs[j], &Ps[j]);
    }
    epilogue_bar();
    const int t = et;
    if (t < T)
        for (int k = 0; k < K; ++k) {
            const int j = chosen[t * kMaxTopK + k];
            if (j >= 0 && j < N) atomicOr(&bits[j * 4 + (t >> 5)], 1u << (t & 31));
        }
    if (et < 32) {   // offsets: lane l scans experts 8l .. 8l+7 (N' <= 256)
        int loc[8], sum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int j = lane * 8 + q;
            const int v = j < N ? (a.pad > 0 ? (hist[j] + a.pad - 1) / a.pad * a.pad : hist[j]) : 0;
            loc[q] = sum;
            sum += v;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int j = lane * 8 + q;
            if (j < N) off[j] = incl - sum + loc[q];
        }
        if (lane == 31) off[N] = incl;
    }
    epilogue_bar();
    for (int j = et; j <= N; j += 128) a.offsets[j] = off[j];
    if (et == 32 && a.losses) balance_losses(a.dims, fs, Ps, a.losses);
    if (a.f_out)
        for (int j = et; j < N; j += 128) {
            a.f_out[j] = fs[j];
            a.P_out[j] = Ps[j];
        }
    if (t < T)
        for (int k = 0; k < K; ++k) {
            int j = chosen[t * kMaxTopK + k];
            j = (j >= 0 && j < N) ? j : 0;
            int rank = __popc(bits[j * 4 + (t >> 5)] & ((1u << (t & 31)) - 1u));
            for (int w = 0; w < (t >> 5); ++w) rank += __popc(bits[j * 4 + w]);
            const int row = off[j] + rank;
            a.perm_slot[(size_t)t * K + k] = row;
            a.perm_token[row] = t;
        }
}

// Routing of the 128 tokens of a tile by the four epilogue warps (thread = token): softmax over
// the N' routed experts, top-K' by logit (lower index on ties), gates, the tile histogram and the
// tile's per-expert affinity sums. `zc` ([n_pad][128] floats, column j of row r at j * 128 + r,
// conflict-free per warp) receives the biased logits and then the exponentials, so TMEM is read
// once and every exponential is computed once.
template <int KMAX>
__device__ __forceinline__ void route_tile(const RouterArgs& a, uint32_t tmem_lanes, float* zc,
                                          int tile, int quarter, int lane, float* colsum,
                                          int* hist, const float* bias_s, int* chosen) {
    const int N = a.N, K = a.K;
    const int row = quarter * 32 + lane;
    const int t = tile * RBM + row;
    const bool valid = t < a.T;
    const int n_chunks = a.n_pad / 32;
    // the other CTAs of the cluster keep their partial logits at the same offset as zc
    const uint32_t part = ptx::smem_addr(zc);
    // pass 1 (TMEM): biased logits, their maximum and the top list
    float zmax = -INFINITY;
    TopK<KMAX> top;
    top.init();
    for (int c = 0; c < n_chunks; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tmem_lanes + c * 32, v);
        ptx::tmem_ld_wait();
        for (int r = 1; r < a.csize; ++r) {   // partial sums of the later K slices, in rank order
            const uint32_t peer = ptx::mapa(part, (uint32_t)r);
            float pv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                pv[i] = ptx::ld_cluster_f32(peer + (uint32_t)(((c * 32 + i) * RBM + row) * 4));
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + pv[i]);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int j = c * 32 + i;
            if (j < N) {
                const float z = __uint_as_float(v[i]) + bias_s[j];
                zc[j * RBM + row] = z;
                zmax = fmaxf(zmax, z);
                top.push(z, j);
            }
        }
    }
    // pass 2: exponentials and the softmax denominator
    float sum = 0.f;
    for (int j = 0; j < N; ++j) {
        const float e = __expf(zc[j * RBM + row] - zmax);
        zc[j * RBM + row] = e;
        sum += e;
    }
    const float inv = 1.0f / sum;
    if (valid) {
        const int q0 = a.skip;   // chosen ranks: q0 .. q0+K'-1
        float gsum = 0.f;
#pragma unroll
        for (int q = 0; q < KMAX; ++q)
            if (q >= q0 && q < q0 + K) gsum += __expf(top.v[q] - zmax) * inv;
        bool bad = !(zmax < INFINITY);
#pragma unroll
        for (int q = 0; q < KMAX; ++q) {
            if (q >= q0 && q < q0 + K) {
                int j = top.i[q];
                if (j < 0) {
                    bad = true;
                    j = 0;
                }
                const float s = __expf(top.v[q] - zmax) * inv;
                a.topk_idx[(size_t)t * K + q - q0] = j;
                a.topk_gate[(size_t)t * K + q - q0] = a.renorm ? s / gsum : s;
                chosen[row * kMaxTopK + q - q0] = j;   // for the one-tile tables
                atomicAdd(&hist[j], 1);
            }
        }
        if (bad) set_status(a.status, MOE_ERR_CORRUPT_INPUT);
    }
    // pass 3: affinities, summed over this warp's 32 tokens per expert column
    for (int c = 0; c < n_chunks; ++c) {
        float s[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int j = c * 32 + i;
            s[i] = (valid && j < N) ? zc[j * RBM + row] * inv : 0.f;
        }
        const float col = column_sums(s, lane);
        colsum[quarter * kMaxRouted + c * 32 + lane] = col;
    }
}

// Backward of the router for the tile's tokens (thread = token): with s = softmax(z) recomputed,
// ds_j = aux_j + (gradient of the chosen gates through g = s or g = s / S), aux_j being the
// balance-loss term (a1 f_j + a2 f'_group(j)) / T, and dz_j = s_j (ds_j - sum_m s_m ds_m).
// dz is written as bf16 [T, n_pad] (zero past N'); its per-tile column sums (for the bias
// gradient) go through the same fixed-order warp reduction as the affinity sums.
__device__ __forceinline__ void route_tile_bwd(const RouterArgs& a, uint32_t tmem_lanes, float* zc,
                                              int tile, int quarter, int lane, float* colsum,
                                              const float* bias_s, const float* aux_s) {
    const int N = a.N, K = a.K;
    const int row = quarter * 32 + lane;
    const int t = tile * RBM + row;
    const bool valid = t < a.T;
    const int n_chunks = a.n_pad / 32;
    float zmax = -INFINITY;
    for (int c = 0; c < n_chunks; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tmem_lanes + c * 32, v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int j = c * 32 + i;
            if (j < N) {
                const float z = __uint_as_float(v[i]) + bias_s[j];
                zc[j * RBM + row] = z;
                zmax = fmaxf(zmax, z);
            }
        }
    }
    float sum = 0.f;
    for (int j = 0; j < N; ++j) {
        const float e = __expf(zc[j * RBM + row] - zmax);
        zc[j * RBM + row] = e;
        sum += e;
    }
    const float inv = 1.0f / sum;
    // chosen experts and the gradient of their gates with respect to their affinities
    int cj[kMaxTopK];
    float cs[kMaxTopK], cd[kMaxTopK];
    float S = 0.f, w = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
        cj[k] = 0;
        cs[k] = 0.f;
        cd[k] = 0.f;
        if (k < K && valid) {
            int j = a.topk_idx[(size_t)t * K + k];
            j = (j >= 0 && j < N) ? j : 0;
            cj[k] = j;
            cs[k] = zc[j * RBM + row] * inv;
            cd[k] = a.dgate[(size_t)t * K + k];
            S += cs[k];
            w += cd[k] * cs[k];
        }
    }
    float sds = 0.f;
    for (int j = 0; j < N; ++j) sds += zc[j * RBM + row] * inv * aux_s[j];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
        if (k < K && valid) {
            cd[k] = a.renorm ? cd[k] / S - w / (S * S) : cd[k];   // chosen part of ds
            sds += cs[k] * cd[k];
        }
    }
    for (int j = 0; j < N; ++j) {
        const float sj = zc[j * RBM + row] * inv;
        zc[j * RBM + row] = valid ? sj * (aux_s[j] - sds) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k)
        if (k < K && valid) zc[cj[k] * RBM + row] += cs[k] * cd[k];
    for (int c = 0; c < n_chunks; ++c) {
        float g[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int j = c * 32 + i;
            g[i] = j < N ? zc[j * RBM + row] : 0.f;
        }
        if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(a.dz + (size_t)t * a.n_pad + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 o;
                __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    o2[h] = __floats2bfloat162_rn(g[8 * q + 2 * h], g[8 * q + 2 * h + 1]);
                dst[q] = o;
            }
        }
        const float col = column_sums(g, lane);
        colsum[quarter * kMaxRouted + c * 32 + lane] = col;
    }
}

template <int KMAX, bool BWD>
__global__ void __launch_bounds__(kThreads, 1) router_tc_kernel(const __grid_constant__ RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring = a.stages * a.stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + ring);
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;
    uint64_t* drain = tfull + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* colsum = reinterpret_cast<float*>(tmem_holder + 4);   // [4][kMaxRouted]
    int* hist = reinterpret_cast<int*>(colsum + 4 * kMaxRouted);  // [kMaxRouted]
    float* bias_s = reinterpret_cast<float*>(hist + kMaxRouted);  // [kMaxRouted]
    float* aux_s = bias_s + kMaxRouted;                           // [kMaxRouted] (backward)
    int* chosen = reinterpret_cast<int*>(aux_s + kMaxRouted);     // [128][kMaxTopK]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int crank = a.csize > 1 ? (int)ptx::cluster_ctarank() : 0;
    const bool leader = crank == 0;
    const int tile = blockIdx.x / a.csize;
    const int n_tiles = gridDim.x / a.csize;
    const int kb_begin = crank * a.k_blocks / a.csize;
    const int kb_end = (crank + 1) * a.k_blocks / a.csize;
    const int N = a.N;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(tfull), 1);
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    for (int j = threadIdx.x; j < kMaxRouted; j += blockDim.x) hist[j] = 0;
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&a.a);
        ptx::prefetch_tmap(&a.b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), a.tmem_cols);
        ptx::tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    for (int j = threadIdx.x; j < kMaxRouted; j += blockDim.x)
        bias_s[j] = (a.bias && j < N) ? a.bias[j] : 0.f;
    if constexpr (BWD) {   // balance-loss gradient per expert: (a1 f_j + a2 f'_group(j)) / T
        const float Tf = (float)a.T, scale = (float)N / ((float)a.K * Tf);
        const int gbase = N / a.D, extra = N % a.D;
        for (int j = threadIdx.x; j < N; j += blockDim.x) {
            const int g = j < extra * (gbase + 1) ? j / (gbase + 1)
                                                  : extra + (j - extra * (gbase + 1)) / gbase;
            const int first = g * gbase + (g < extra ? g : extra);
            const int size = gbase + (g < extra ? 1 : 0);
            float fs = 0.f;
            for (int q = first; q < first + size; ++q) fs += scale * (float)a.counts[q];
            aux_s[j] = (a.a1 * scale * (float)a.counts[j] + a.a2 * fs / (float)size) / Tf;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int kb = kb_begin; kb < kb_end; ++kb) {
                if (!wait_phase(ptx::smem_addr(&empty[stage]), phase ^ 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = ptx::smem_addr(&full[stage]);
                uint8_t* st = base + stage * a.stage_bytes;
                ptx::mbar_arrive_expect_tx(fb, a.stage_bytes);
                ptx::tma_load_2d(ptx::smem_addr(st), &a.a, kb * RBK, tile * RBM, fb);
                ptx::tma_load_2d(ptx::smem_addr(st + RBM * RBK * 2), &a.b, kb * RBK, 0, fb);
                ++issued;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) {
                for (int i = 0; i < issued && i < a.stages; ++i) {
                    if (--stage < 0) {
                        stage = a.stages - 1;
                        phase ^= 1;
                    }
                    drain_wait(ptx::smem_addr(&full[stage]), phase);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(RBM, a.n_pad);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, any = false;
            for (int kb = kb_begin; kb < kb_end; ++kb) {
                if (!wait_phase(ptx::smem_addr(&full[stage]), phase, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t a0 = ptx::smem_addr(base + stage * a.stage_bytes);
                const uint32_t b0 = a0 + RBM * RBK * 2;
#pragma unroll
                for (int k = 0; k < RBK / 16; ++k)
                    ptx::mma_f16(tmem, ptx::sw128_kmajor_desc(a0 + k * 32),
                                 ptx::sw128_kmajor_desc(b0 + k * 32), idesc,
                                 (kb != kb_begin || k != 0) ? 1u : 0u);
                any = true;
                ptx::mma_commit(ptx::smem_addr(&empty[stage]));
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (ok) ptx::mma_commit(ptx::smem_addr(tfull));
            else if (any) {
                ptx::mma_commit(ptx::smem_addr(drain));
                drain_wait(ptx::smem_addr(drain), 0);
            }
        }
    } else if (!leader) {
        // ------------------------------------------- partial logits of a later K slice ----
        // kept in the idle ring as [n_pad][128] floats for the first CTA of the cluster
        const int quarter = warp & 3;
        int ok = 1;
        if (lane == 0) ok = wait_phase(ptx::smem_addr(tfull), 0, abort_flag, a.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        float* part = reinterpret_cast<float*>(base);
        const int row = quarter * 32 + lane;
        if (ok) ptx::tc_fence_after();
        for (int c = 0; c < a.n_pad / 32; ++c) {
            uint32_t v[32];
            if (ok) {
                ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + c * 32, v);
                ptx::tmem_ld_wait();
            }
#pragma unroll
            for (int i = 0; i < 32; ++i)   // zeros if this CTA gave up (its status is set)
                part[(c * 32 + i) * RBM + row] = ok ? __uint_as_float(v[i]) : 0.f;
        }
    }
    if (a.csize > 1) {   // the partial logits are in place; every thread of the cluster
        __syncwarp();
        ptx::cluster_sync();
    }
    if (warp >= 2 && leader) {
        // --------------------------------------------------------------------- epilogue ----
        const int quarter = warp & 3;
        const int et = threadIdx.x - 64;   // 0..127 over the four epilogue warps
        int ok = 1;
        if (lane == 0) ok = wait_phase(ptx::smem_addr(tfull), 0, abort_flag, a.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16);
        bool routed_here = false;
        if (ok) {
            ptx::tc_fence_after();
            // the MMAs are complete, so the TMA ring is idle and holds the per-token logit rows
            if constexpr (BWD)
                route_tile_bwd(a, tb, reinterpret_cast<float*>(base), tile, quarter, lane, colsum,
                               bias_s, aux_s);
            else
                route_tile<KMAX>(a, tb, reinterpret_cast<float*>(base), tile, quarter, lane,
                                 colsum, hist, bias_s, chosen);
            routed_here = true;
        }
        ptx::tc_fence_before();
        epilogue_bar();
        if (routed_here) {
            for (int j = et; j < N; j += 128) {
                const float col = ((colsum[j] + colsum[kMaxRouted + j]) +
                                   colsum[2 * kMaxRouted + j]) + colsum[3 * kMaxRouted + j];
                if constexpr (BWD) {
                    a.tile_dz[(size_t)j * n_tiles + tile] = col;
                } else {
                    a.tile_psum[(size_t)j * n_tiles + tile] = col;
                    a.tile_counts[(size_t)j * n_tiles + tile] = hist[j];
                }
            }
        }
        if constexpr (!BWD) {
            if (a.fused) finish_single_tile(a, base, hist, colsum, chosen, et, lane);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (a.csize > 1) ptx::cluster_sync();   // the first CTA has read the others' partial logits
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, a.tmem_cols);
    }
}

}  // namespace

static cudaError_t router_args(const Dims& m, const void* u, const void* centroids,
                               const float* bias, RouterArgs& a) {
    a.n_pad = router_npad(m);
    if (!encode_bf16_map(&a.a, u, (uint64_t)m.T, (uint64_t)m.d, RBM) ||
        !encode_bf16_map(&a.b, centroids, (uint64_t)m.N, (uint64_t)m.d, a.n_pad))
        return cudaErrorInvalidValue;
    a.bias = bias;
    a.dims = m;
    a.T = m.T;
    a.N = m.N;
    a.K = m.K;
    a.renorm = m.renorm;
    a.skip = m.skip;
    a.k_blocks = m.d / RBK;
    a.stage_bytes = (uint32_t)(RBM * RBK * 2 + a.n_pad * RBK * 2);
    a.stages = (int)std::min<uint32_t>(kMaxStages, (192u * 1024u) / a.stage_bytes);
    int cols = 32;
    while (cols < a.n_pad) cols *= 2;
    a.tmem_cols = cols;
    // few tiles: up to 8 CTAs per tile, while the grid stays within one wave and every CTA keeps
    // at least two K blocks
    const int n_tiles = (m.T + RBM - 1) / RBM;
    int c = 1;
    while (c < 8 && (long)n_tiles * c * 2 <= sm_count() && a.k_blocks / (c * 2) >= 2) c *= 2;
    a.csize = c;
    return cudaSuccess;
}

template <int KMAX, bool BWD>
static cudaError_t launch_router_kernel(const Dims& m, const RouterArgs& a, cudaStream_t st) {
    const size_t smem = 1024 + (size_t)a.stages * a.stage_bytes + 8 * (2 * kMaxStages + 2) + 16 +
                        4 * (4 * kMaxRouted + 3 * kMaxRouted) + 4 * RBM * kMaxTopK;
    const int n_tiles = (m.T + RBM - 1) / RBM;
    auto kern = router_tc_kernel<KMAX, BWD>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    if (a.csize == 1) {
        e = launch_pdl(kern, dim3(n_tiles), dim3(kThreads), smem, st, a);
    } else {   // clusters of csize CTAs per tile
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(n_tiles * a.csize);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)a.csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kern, a);
    }
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_router_tc(const Dims& m, const void* u, const void* centroids,
                             const float* bias, int* topk_idx, float* topk_gate, int* tile_counts,
                             float* tile_psum, int* status, cudaStream_t st,
                             const SingleTileTables* tables) {
    RouterArgs a{};
    cudaError_t e = router_args(m, u, centroids, bias, a);
    if (e != cudaSuccess) return e;
    a.topk_idx = topk_idx;
    a.topk_gate = topk_gate;
    a.tile_counts = tile_counts;
    a.tile_psum = tile_psum;
    a.status = status;
    if (tables) {
        if (m.T > RBM) return cudaErrorInvalidValue;   // one tile only
        a.fused = 1;
        a.pad = tables->pad;
        a.counts_out = tables->counts;
        a.psum_out = tables->psum;
        a.offsets = tables->offsets;
        a.perm_token = tables->perm_token;
        a.perm_slot = tables->perm_slot;
        a.f_out = tables->f;
        a.P_out = tables->P;
        a.losses = tables->losses;
    }
    return m.skip + m.K <= 8 ? launch_router_kernel<8, false>(m, a, st)
                             : launch_router_kernel<16, false>(m, a, st);
}

cudaError_t launch_router_bwd(const Dims& m, const void* u, const void* centroids,
                              const float* bias, const int* topk_idx, const float* dgate,
                              const int* counts, void* dz, float* tile_dz, int* status,
                              cudaStream_t st) {
    if (m.T == 0) return cudaSuccess;
    RouterArgs a{};
    cudaError_t e = router_args(m, u, centroids, bias, a);
    if (e != cudaSuccess) return e;
    a.topk_idx = const_cast<int*>(topk_idx);
    a.csize = 1;   // the backward epilogue needs the whole logit row of a token in one CTA
    a.dgate = dgate;
    a.counts = counts;
    a.dz = static_cast<__nv_bfloat16*>(dz);
    a.tile_dz = tile_dz;
    a.a1 = m.a1;
    a.a2 = m.a2;
    a.D = m.D;
    a.status = status;
    return launch_router_kernel<8, true>(m, a, st);
}

}  // namespace moe
