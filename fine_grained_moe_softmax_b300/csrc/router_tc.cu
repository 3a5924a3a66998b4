// router_tc.cu -- router of bf16 layers on the tensor cores.
//
// [P1] "DeepSeekMoE 论文解读" (xxmr.cn), §方法细节: gates come from Topk({s_{j,t}}, mK) over the
//      routed experts (the K_s shared experts are always active and are not ranked).
// [P2] "【论文总结】MoE" (mickeyding.github.io), §2.2: s_{j,t} = softmax_j(u_t . e_j) against the
//      learnable centroids e_j; §2.3: f_i counts selections, P_i averages s over the T tokens.
//
// The logits of a 128-token tile are one [128 x d] x [d x N'] product: the tile's token rows and
// the centroids stream through a TMA ring into tcgen05.mma (M = 128, N = N' rounded up to 32),
// accumulating fp32 logits in TMEM. A ring stage holds up to four 64-deep K chunks, and each
// operand of a stage is one 3D tensor copy (a copy costs about the same whatever its size, so
// fewer, larger copies move more bytes per cycle). When there are few tiles (decode-sized
// batches), a cluster of C CTAs shares a tile, each over 1/C of d; the other CTAs leave their
// partial logits in their shared memory and the first adds them to its own, in rank order,
// through distributed shared memory, so the sum does not depend on timing. The other CTAs exit
// once the first CTA's threads have read them (a split cluster barrier).
//
// Sixteen epilogue warps route the tile: four per TMEM lane quarter (warp w reads lanes
// 32*(w%4) .. +31), each over a quarter of the expert columns. A thread owns one token of one
// column slice: it reads the slice's logits from TMEM once, adds the optional bias, keeps them in
// the (by then idle) TMA ring, and keeps the slice's maximum and its top list (ranked by logit, the
// lower index first on ties). The slices' maxima give the softmax shift, their exponential sums
// (added in slice order) the denominator, and a shuffle transpose the tile's per-expert sums of
// affinities in a fixed order. The four slice lists of a token are merged by four lanes, one list
// each, in K' rounds of a 4-way maximum whose ties go to the lower slice (the lower indices);
// those lanes then write the token's experts and gates and count the tile's histogram. The
// epilogue runs once per launch and its instructions are fetched cold, so it is one non-inlined
// function with rolled loops; warps whose 32 tokens are all past the batch skip its phases.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "waits.cuh"

namespace moe {

namespace {

constexpr int RBM = 128;
constexpr int RBK = 64;
constexpr int kEpiWarpsBwd = 4;                        // backward: one warp per lane quarter
constexpr int kEpiWarpsFwd = 16;                       // forward: four per lane quarter
constexpr int kMaxStages = 8;

__host__ __device__ constexpr int router_threads(bool bwd) {
    return 64 + 32 * (bwd ? kEpiWarpsBwd : kEpiWarpsFwd);
}

// Scalar arguments of the router kernel. Kernel code reads them from a copy in shared memory (or
// from registers): the kernel takes the tensor maps' addresses, which makes every direct read of
// a kernel argument a generic load of the argument buffer, and the mbarrier waits' memory
// clobbers would otherwise force such a reload on every pipeline step.
struct RouterParams {
    const float* bias;    // [N'] or null
    int T, N, K, renorm, skip, k_blocks, n_pad, stages, tmem_cols;
    int kc;               // 64-deep K chunks per stage (one tensor copy each for u and centroids)
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

struct RouterArgs {
    CUtensorMap a;        // u [T, d] in 64-column chunks, box [kc x 128 x 64]
    CUtensorMap b;        // centroids [N', d] in 64-column chunks, box [kc x n_pad x 64]
    RouterParams p;
};
static_assert(sizeof(RouterParams) % 8 == 0, "copied in 4-byte words");

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

// One halving step with the shuffle partner at lane distance MASK: lanes with `upper` clear keep
// columns [0, HALF) and receive the partner's, lanes with it set keep [HALF, 2*HALF).
template <int HALF, int MASK>
__device__ __forceinline__ void halve_x(float (&v)[8], bool upper) {
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
        const float send = upper ? v[i] : v[i + HALF];
        const float keep = upper ? v[i + HALF] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
    }
}

// After this, lane l of the warp holds the sum over the 32 lanes of column (l >> 2) & 7 of
// v[0..7] (lanes 4c .. 4c+3 hold column c), added in one fixed pattern.
__device__ __forceinline__ float column_sums8(float (&v)[8], int lane) {
    halve_x<4, 16>(v, lane & 16);
    halve_x<2, 8>(v, lane & 8);
    halve_x<1, 4>(v, lane & 4);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    return v[0];
}

template <int THREADS>
__device__ __forceinline__ void epilogue_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
}

// Barrier of the epilogue warps that also returns 1 only if v != 0 in every one of their threads.
template <int THREADS>
__device__ __forceinline__ int epilogue_and(int v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v), "n"(THREADS)
        : "memory");
    return r;
}

// The routing tables of a one-tile batch, by the sixteen epilogue warps (et = 0..511) after the
// tile is routed: totals, offsets (exclusive scan, segments padded to a.pad), the balance
// statistics and the stable permutation. The rank of token t in expert j is the number of earlier
// tokens of the tile choosing j (a prefix popcount of j's token bitmap); these are the results of
// the finalize and scatter kernels for the same batch, bit for bit. `scratch` is the idle TMA
// ring. Every epilogue warp runs the whole sequence (the barriers need all of them).
constexpr int kEpiThreadsFwd = 32 * kEpiWarpsFwd;

__device__ __noinline__ void finish_single_tile(const RouterParams& a, uint8_t* scratch,
                                                const int* hist, const float* colsum,
                                                const int* chosen, int et) {
    const int N = a.N, K = a.K, T = a.T, lane = et & 31;
    uint32_t* bits = reinterpret_cast<uint32_t*>(scratch);         // [N'][4]: tokens 0..127
    int* off = reinterpret_cast<int*>(bits + 4 * kMaxRouted);       // [N' + 1]
    float* ptot = reinterpret_cast<float*>(off + kMaxRouted + 1);   // [N']
    float* fs = ptot + kMaxRouted;                                  // [N']
    float* Ps = fs + kMaxRouted;                                    // [N']
    int* seg = reinterpret_cast<int*>(Ps + kMaxRouted);             // [N']: padded segment rows
    const int pad = a.pad;
    for (int i = et; i < 4 * N; i += kEpiThreadsFwd) bits[i] = 0u;
    for (int j = et; j < N; j += kEpiThreadsFwd) {
        const float col = ((colsum[j] + colsum[kMaxRouted + j]) + colsum[2 * kMaxRouted + j]) +
                          colsum[3 * kMaxRouted + j];
        seg[j] = pad > 0 ? (hist[j] + pad - 1) / pad * pad : hist[j];
        ptot[j] = col;
        a.counts_out[j] = hist[j];
        a.psum_out[j] = col;
        balance_fp(a.dims, hist[j], col, &fs[j], &Ps[j]);
    }
    epilogue_bar<kEpiThreadsFwd>();
    for (int x = et; x < T * K; x += kEpiThreadsFwd) {
        const int t = x / K, j = chosen[t * kMaxTopK + x % K];
        if (j >= 0 && j < N) atomicOr(&bits[j * 4 + (t >> 5)], 1u << (t & 31));
    }
    if (et < 32) {   // offsets: lane l scans experts 8l .. 8l+7 (N' <= 256)
        int sum = 0;
#pragma unroll 1
        for (int j = lane * 8; j < min(lane * 8 + 8, N); ++j) sum += seg[j];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - sum;
#pragma unroll 1
        for (int j = lane * 8; j < min(lane * 8 + 8, N); ++j) {
            off[j] = run;
            run += seg[j];
        }
        if (lane == 31) off[N] = incl;
    }
    epilogue_bar<kEpiThreadsFwd>();
    // the balance losses by the last warp, beside the permutation below (a decode-sized batch
    // leaves that warp without permutation entries)
    if (et >= kEpiThreadsFwd - 32 && a.losses) balance_losses_warp(a.dims, fs, Ps, a.losses, lane);
    for (int j = et; j <= N; j += kEpiThreadsFwd) a.offsets[j] = off[j];
    if (a.f_out)
        for (int j = et; j < N; j += kEpiThreadsFwd) {
            a.f_out[j] = fs[j];
            a.P_out[j] = Ps[j];
        }
    for (int x = et; x < T * K; x += kEpiThreadsFwd) {
        const int t = x / K;
        int j = chosen[t * kMaxTopK + x % K];
        j = (j >= 0 && j < N) ? j : 0;
        int rank = __popc(bits[j * 4 + (t >> 5)] & ((1u << (t & 31)) - 1u));
        for (int w = 0; w < (t >> 5); ++w) rank += __popc(bits[j * 4 + w]);
        const int row = off[j] + rank;
        a.perm_slot[x] = row;
        a.perm_token[row] = t;
    }
}

// Routing of the tile's tokens by the sixteen epilogue warps. Warp w (2 <= w < 18) reads TMEM lane
// quarter q = w % 4 (tokens 32q .. 32q+31) and column slice h = (w - 2) / 4 of n_pad / 4 columns.
// Shared scratch: zc = [n_pad][128] floats at the start of the idle ring (column j of token row r
// at j * 128 + r, conflict-free per warp), then the slice lists [4][KMAX][128] (values, then
// indices); `red` holds the slices' maxima and exponential sums [2][4][128].
template <int KMAX>
__device__ __noinline__ void route_tile(const RouterParams& a, uint32_t tmem, uint8_t* ring,
                                        int tile, int warp, int lane, float* colsum, int* hist,
                                        const float* bias_s, int* chosen, float* chosen_s,
                                        float* red) {
    const int N = a.N, K = a.K;
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const int rows_valid = min(RBM, a.T - tile * RBM);
    const bool valid = row < rows_valid;
    const int cs = a.n_pad >> 2;   // columns per slice, a multiple of 8
    const int c0 = h * cs;
    float* zc = reinterpret_cast<float*>(ring);
    float* lv = zc + a.n_pad * RBM;
    int* li = reinterpret_cast<int*>(lv + 4 * KMAX * RBM);
    float* red_max = red;
    float* red_sum = red + 4 * RBM;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    // the other CTAs of the cluster keep their partial logits at the same offset as zc
    const uint32_t part = ptx::smem_addr(zc);
    // a warp whose 32 rows are all past the batch (in a tile of at most 96 tokens) skips phases
    // A, B and D and contributes zero column sums, leaving the issue slots to the warps with tokens
    const bool qvalid = q * 32 < rows_valid;

    // A: the slice's biased logits, their maximum and the slice's top list. The epilogue runs once
    // per launch, so its code is fetched cold: loops stay rolled where unrolling buys nothing.
    float mloc = -INFINITY;
    TopK<KMAX> top;
    top.init();
#pragma unroll 1
    for (int c = c0; c < (qvalid ? c0 + cs : c0); c += 8) {
        uint32_t v[8];
        ptx::tmem_ld_32x32b_x8(tl + c, v);
        ptx::tmem_ld_wait();
        if (valid && a.csize > 1) {
            // partial sums of the later K slices, added in rank order; the loads of all the
            // cluster's CTAs for four columns are issued before any of them is used
#pragma unroll
            for (int h4 = 0; h4 < 8; h4 += 4) {
                float pv[7][4];
#pragma unroll
                for (int r = 1; r < 8; ++r)
                    if (r < a.csize) {
                        const uint32_t peer = ptx::mapa(part, (uint32_t)r);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            pv[r - 1][i] = ptx::ld_cluster_f32(
                                peer + (uint32_t)(((c + h4 + i) * RBM + row) * 4));
                    }
#pragma unroll
                for (int r = 1; r < 8; ++r)
                    if (r < a.csize) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            v[h4 + i] = __float_as_uint(__uint_as_float(v[h4 + i]) + pv[r - 1][i]);
                    }
            }
        }
        // bias_s holds zeros past N', so the padding columns keep their (unused) raw values
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int j = c + i;
            const float z = __uint_as_float(v[i]) + bias_s[j];
            zc[j * RBM + row] = z;
            if (j < N) {
                mloc = fmaxf(mloc, z);
                top.push(z, j);
            }
        }
    }
    red_max[h * RBM + row] = mloc;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        lv[(h * KMAX + k) * RBM + row] = top.v[k];
        li[(h * KMAX + k) * RBM + row] = top.i[k];
    }
    epilogue_bar<kEpiThreadsFwd>();

    // B: exponentials of the slice and its part of the softmax denominator
    const float zmax = fmaxf(fmaxf(red_max[row], red_max[RBM + row]),
                             fmaxf(red_max[2 * RBM + row], red_max[3 * RBM + row]));
    float ssum = 0.f;
    const int c1 = qvalid ? min(c0 + cs, N) : c0;
    for (int j = c0; j < c1; ++j) {
        const float e = __expf(zc[j * RBM + row] - zmax);
        zc[j * RBM + row] = e;
        ssum += e;
    }
    red_sum[h * RBM + row] = ssum;
    epilogue_bar<kEpiThreadsFwd>();

    // C: the slice's affinities summed over the warp's 32 tokens, per expert column
    {
        const float inv = 1.0f / (((red_sum[row] + red_sum[RBM + row]) + red_sum[2 * RBM + row]) +
                                  red_sum[3 * RBM + row]);
        for (int c = c0; c < c0 + cs; c += 8) {
            float sv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = c + i;
                sv[i] = (valid && j < N) ? zc[j * RBM + row] * inv : 0.f;
            }
            const float col = column_sums8(sv, lane);
            if ((lane & 3) == 0) colsum[q * kMaxRouted + c + (lane >> 2)] = col;
        }
    }

    // D: merge of the token's four slice lists by four lanes (lane & 3 = the list it reads), one
    // rank per round; the chosen ranks' experts and affinities go to `chosen` / `chosen_s`
    {
        const int tr = q * 32 + h * 8 + (lane >> 2);
        const int sub = lane & 3;
        const bool tvalid = tr < rows_valid;
        const float zm = fmaxf(fmaxf(red_max[tr], red_max[RBM + tr]),
                               fmaxf(red_max[2 * RBM + tr], red_max[3 * RBM + tr]));
        const float tinv = 1.0f / (((red_sum[tr] + red_sum[RBM + tr]) + red_sum[2 * RBM + tr]) +
                                   red_sum[3 * RBM + tr]);
        const int q0 = a.skip;   // chosen ranks: q0 .. q0+K'-1
        int p = 0;
        float gsum = 0.f;
        bool bad = !(zm < INFINITY);
#pragma unroll 1
        for (int r = 0; r < (qvalid ? q0 + K : 0); ++r) {
            float v = p < KMAX ? lv[(sub * KMAX + p) * RBM + tr] : -INFINITY;
            int ix = p < KMAX ? li[(sub * KMAX + p) * RBM + tr] : -1;
            int sl = sub;
#pragma unroll
            for (int m = 1; m <= 2; m <<= 1) {   // 4-way maximum; ties to the lower slice
                const float ov = __shfl_xor_sync(0xffffffffu, v, m);
                const int oi = __shfl_xor_sync(0xffffffffu, ix, m);
                const int os = __shfl_xor_sync(0xffffffffu, sl, m);
                if (ov > v || (ov == v && os < sl)) {
                    v = ov;
                    ix = oi;
                    sl = os;
                }
            }
            if (sl == sub) ++p;
            if (r >= q0) {
                const float sj = __expf(v - zm) * tinv;
                gsum += sj;
                if (ix < 0) {
                    bad = true;
                    ix = 0;
                }
                if (sub == 0) {
                    chosen[tr * kMaxTopK + r - q0] = ix;   // also for the one-tile tables
                    chosen_s[tr * kMaxTopK + r - q0] = sj;
                }
            }
        }
        __syncwarp();
        if (tvalid) {
            const int t = tile * RBM + tr;
#pragma unroll 1
            for (int k = sub; k < K; k += 4) {
                const int j = chosen[tr * kMaxTopK + k];
                const float sj = chosen_s[tr * kMaxTopK + k];
                a.topk_idx[(size_t)t * K + k] = j;
                a.topk_gate[(size_t)t * K + k] = a.renorm ? sj / gsum : sj;
                atomicAdd(&hist[j], 1);
            }
            if (bad && sub == 0) set_status(a.status, MOE_ERR_CORRUPT_INPUT);
        }
    }
}

// Backward of the router for the tile's tokens (thread = token): with s = softmax(z) recomputed,
// ds_j = aux_j + (gradient of the chosen gates through g = s or g = s / S), aux_j being the
// balance-loss term (a1 f_j + a2 f'_group(j)) / T, and dz_j = s_j (ds_j - sum_m s_m ds_m).
// dz is written as bf16 [T, n_pad] (zero past N'); its per-tile column sums (for the bias
// gradient) go through the same fixed-order warp reduction as the affinity sums.
__device__ __forceinline__ void route_tile_bwd(const RouterParams& a, uint32_t tmem_lanes, float* zc,
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
__global__ void __launch_bounds__(router_threads(BWD), 1)
    router_tc_kernel(const __grid_constant__ RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // scalars read once into registers (the copy in shared memory serves the epilogue)
    const int stages = a.p.stages, csize = a.p.csize, k_blocks = a.p.k_blocks, N = a.p.N;
    const int kc = a.p.kc;
    const uint32_t stage_bytes = a.p.stage_bytes;
    int* const status = a.p.status;
    const uint32_t ring = stages * stage_bytes;
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
    float* chosen_s = reinterpret_cast<float*>(chosen + RBM * kMaxTopK);   // [128][kMaxTopK]
    float* red = chosen_s + RBM * kMaxTopK;                               // [2][4][128] (forward)
    RouterParams* ps = reinterpret_cast<RouterParams*>(red + 2 * 4 * RBM);   // the scalars

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int crank = csize > 1 ? (int)ptx::cluster_ctarank() : 0;
    const bool leader = crank == 0;
    const int tile = blockIdx.x / csize;
    const int n_tiles = gridDim.x / csize;
    const int kb_begin = crank * k_blocks / csize;
    const int kb_end = (crank + 1) * k_blocks / csize;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
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
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), a.p.tmem_cols);
        ptx::tmem_relinquish();
    }
    if (warp == 2) {   // the epilogue's copy of the scalars (ordered by the epilogue's barriers)
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&a.p);
        uint32_t* dst = reinterpret_cast<uint32_t*>(ps);
        for (int i = lane; i < (int)(sizeof(RouterParams) / 4); i += 32) dst[i] = src[i];
    }
    pdl_wait();
    pdl_trigger();
    // the producer thread initialised the barriers itself: it issues the ring's first stages
    // before the block-wide sync, so that these loads overlap the TMEM allocation and the rest of
    // the set-up (the ring is fresh, every stage is free)
    int pre_loads = 0;
    if (warp == 0 && lane == 0) {
        for (int kb = kb_begin; kb < kb_end && pre_loads < stages; kb += kc, ++pre_loads) {
            const uint32_t fb = ptx::smem_addr(&full[pre_loads]);
            uint8_t* st = base + pre_loads * stage_bytes;
            ptx::mbar_arrive_expect_tx(fb, stage_bytes);
            ptx::tma_load_3d(ptx::smem_addr(st), &a.a, 0, tile * RBM, kb, fb);
            ptx::tma_load_3d(ptx::smem_addr(st + kc * RBM * RBK * 2), &a.b, 0, 0, kb, fb);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int stage = pre_loads % stages;
            uint32_t phase = pre_loads == stages ? 1u : 0u;
            int issued = pre_loads;
            bool ok = true;
            for (int kb = kb_begin + pre_loads * kc; kb < kb_end; kb += kc) {
                if (!wait_phase(ptx::smem_addr(&empty[stage]), phase ^ 1, abort_flag, status)) {
                    ok = false;
                    break;
                }
                // the boxes always carry kc chunks (their full bytes count, chunks past d are
                // zero-filled); the MMAs use only the chunks below kb_end
                const uint32_t fb = ptx::smem_addr(&full[stage]);
                uint8_t* st = base + stage * stage_bytes;
                ptx::mbar_arrive_expect_tx(fb, stage_bytes);
                ptx::tma_load_3d(ptx::smem_addr(st), &a.a, 0, tile * RBM, kb, fb);
                ptx::tma_load_3d(ptx::smem_addr(st + kc * RBM * RBK * 2), &a.b, 0, 0, kb, fb);
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) {
                for (int i = 0; i < issued && i < stages; ++i) {
                    if (--stage < 0) {
                        stage = stages - 1;
                        phase ^= 1;
                    }
                    drain_wait(ptx::smem_addr(&full[stage]), phase);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(RBM, a.p.n_pad);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, any = false;
            const uint32_t b_chunk = (uint32_t)a.p.n_pad * RBK * 2;
            for (int kb = kb_begin; kb < kb_end; kb += kc) {
                if (!wait_phase(ptx::smem_addr(&full[stage]), phase, abort_flag, status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t a0 = ptx::smem_addr(base + stage * stage_bytes);
                const uint32_t b0 = a0 + kc * RBM * RBK * 2;
                const int nc = min(kc, kb_end - kb);
                for (int c = 0; c < nc; ++c) {
                    const uint32_t ac = a0 + c * RBM * RBK * 2, bc = b0 + c * b_chunk;
#pragma unroll
                    for (int k = 0; k < RBK / 16; ++k)
                        ptx::mma_f16(tmem, ptx::sw128_kmajor_desc(ac + k * 32),
                                     ptx::sw128_kmajor_desc(bc + k * 32), idesc,
                                     (kb != kb_begin || c != 0 || k != 0) ? 1u : 0u);
                }
                any = true;
                ptx::mma_commit(ptx::smem_addr(&empty[stage]));
                if (++stage == stages) {
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
        const int n_pad = a.p.n_pad;
        int ok = 1;
        if (lane == 0) ok = wait_phase(ptx::smem_addr(tfull), 0, abort_flag, status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        float* part = reinterpret_cast<float*>(base);
        const int row = quarter * 32 + lane;
        const int cs = BWD ? n_pad : n_pad >> 2;   // this warp's column slice
        const int c0 = BWD ? 0 : ((warp - 2) >> 2) * cs;
        if (ok) ptx::tc_fence_after();
        for (int c = c0; c < c0 + cs; c += 8) {
            uint32_t v[8];
            if (ok) {
                ptx::tmem_ld_32x32b_x8(tmem + ((uint32_t)(quarter * 32) << 16) + c, v);
                ptx::tmem_ld_wait();
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)   // zeros if this CTA gave up (its status is set)
                part[(c + i) * RBM + row] = ok ? __uint_as_float(v[i]) : 0.f;
        }
    } else {
        // the first CTA's epilogue warps: per-expert inputs of the epilogue, read while the K loop
        // runs (off the producer's path; the epilogue's first barrier publishes them)
        constexpr int kEpi = router_threads(BWD) - 64;
        const int et = threadIdx.x - 64;
        {
            const float* bias = a.p.bias;
            for (int j = et; j < kMaxRouted; j += kEpi)
                bias_s[j] = (bias && j < N) ? bias[j] : 0.f;
        }
        if constexpr (BWD) {   // balance-loss gradient per expert: (a1 f_j + a2 f'_group(j)) / T
            const int* counts = a.p.counts;
            const int K = a.p.K, D = a.p.D;
            const float Tf = (float)a.p.T, scale = (float)N / ((float)K * Tf);
            const float a1 = a.p.a1, a2 = a.p.a2;
            const int gbase = N / D, extra = N % D;
            for (int j = et; j < N; j += kEpi) {
                const int g = j < extra * (gbase + 1) ? j / (gbase + 1)
                                                      : extra + (j - extra * (gbase + 1)) / gbase;
                const int first = g * gbase + (g < extra ? g : extra);
                const int size = gbase + (g < extra ? 1 : 0);
                float fs = 0.f;
                for (int q = first; q < first + size; ++q) fs += scale * (float)counts[q];
                aux_s[j] = (a1 * scale * (float)counts[j] + a2 * fs / (float)size) / Tf;
            }
        }
    }
    if (csize > 1) {   // the partial logits are in place; every thread of the cluster
        __syncwarp();
        ptx::cluster_sync();
        // the first CTA's producer and MMA warps read no partial logits
        if (leader && warp < 2) ptx::cluster_arrive();
    }
    if (warp >= 2 && leader) {
        // --------------------------------------------------------------------- epilogue ----
        constexpr int kEpiThreads = router_threads(BWD) - 64;
        const int quarter = warp & 3;
        const int et = threadIdx.x - 64;   // 0 .. kEpiThreads-1 over the epilogue warps
        int ok = 1;
        if (lane == 0) ok = wait_phase(ptx::smem_addr(tfull), 0, abort_flag, status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // the forward epilogue's barriers need every warp; this barrier also publishes the
        // scalars' copy and the per-expert inputs
        ok = epilogue_and<kEpiThreads>(ok);
        const RouterParams& sp = *ps;
        bool routed_here = false;
        if (ok) {
            ptx::tc_fence_after();
            // the MMAs are complete, so the TMA ring is idle and holds the per-token logit rows
            if constexpr (BWD)
                route_tile_bwd(sp, tmem + ((uint32_t)(quarter * 32) << 16),
                               reinterpret_cast<float*>(base), tile, quarter, lane, colsum,
                               bias_s, aux_s);
            else
                route_tile<KMAX>(sp, tmem, base, tile, warp, lane, colsum, hist, bias_s, chosen,
                                 chosen_s, red);
            routed_here = true;
        }
        if (csize > 1) {   // this thread has read its share of the partial logits
            __syncwarp();
            ptx::cluster_arrive();
        }
        ptx::tc_fence_before();
        epilogue_bar<kEpiThreads>();
        if (routed_here) {
            float* tile_dz = sp.tile_dz;
            float* tile_psum = sp.tile_psum;
            int* tile_counts = sp.tile_counts;
            for (int j = et; j < N; j += kEpiThreads) {
                const float col = ((colsum[j] + colsum[kMaxRouted + j]) +
                                   colsum[2 * kMaxRouted + j]) + colsum[3 * kMaxRouted + j];
                if constexpr (BWD) {
                    tile_dz[(size_t)j * n_tiles + tile] = col;
                } else {
                    tile_psum[(size_t)j * n_tiles + tile] = col;
                    tile_counts[(size_t)j * n_tiles + tile] = hist[j];
                }
            }
        }
        if constexpr (!BWD) {
            if (sp.fused) finish_single_tile(sp, base, hist, colsum, chosen, et);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (csize > 1) {
        // the first CTA's threads arrived once they had read the others' partial logits; the
        // other CTAs keep their shared memory until then
        if (!leader) ptx::cluster_arrive();
        ptx::cluster_wait();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, a.p.tmem_cols);
    }
}

}  // namespace

static cudaError_t router_args(const Dims& m, const void* u, const void* centroids,
                               const float* bias, RouterArgs& a) {
    a.p.n_pad = router_npad(m);
    // a stage of up to 96 KB: kc 64-deep chunks of the u tile and of the centroids, each loaded by
    // one tensor copy (the ring keeps at least two stages)
    const uint32_t chunk_bytes = (uint32_t)(RBM * RBK * 2 + a.p.n_pad * RBK * 2);
    a.p.kc = (int)std::max<uint32_t>(1u, std::min<uint32_t>(4u, (96u * 1024u) / chunk_bytes));
    if (!encode_bf16_map_chunks(&a.a, u, (uint64_t)m.T, (uint64_t)m.d, RBM, a.p.kc) ||
        !encode_bf16_map_chunks(&a.b, centroids, (uint64_t)m.N, (uint64_t)m.d, a.p.n_pad, a.p.kc))
        return cudaErrorInvalidValue;
    a.p.bias = bias;
    a.p.dims = m;
    a.p.T = m.T;
    a.p.N = m.N;
    a.p.K = m.K;
    a.p.renorm = m.renorm;
    a.p.skip = m.skip;
    a.p.k_blocks = m.d / RBK;
    a.p.stage_bytes = chunk_bytes * (uint32_t)a.p.kc;
    a.p.stages = (int)std::min<uint32_t>(kMaxStages, (192u * 1024u) / a.p.stage_bytes);
    int cols = 32;
    while (cols < a.p.n_pad) cols *= 2;
    a.p.tmem_cols = cols;
    // few tiles: up to 8 CTAs per tile, while the grid stays within one wave and every CTA keeps
    // at least two K blocks
    const int n_tiles = (m.T + RBM - 1) / RBM;
    int c = 1;
    while (c < 8 && (long)n_tiles * c * 2 <= sm_count() && a.p.k_blocks / (c * 2) >= 2) c *= 2;
    a.p.csize = c;
    return cudaSuccess;
}

template <int KMAX, bool BWD>
static cudaError_t launch_router_kernel(const Dims& m, const RouterArgs& a, cudaStream_t st) {
    const size_t smem = 1024 + (size_t)a.p.stages * a.p.stage_bytes + 8 * (2 * kMaxStages + 2) + 16 +
                        4 * (4 * kMaxRouted + 3 * kMaxRouted) + 2 * 4 * RBM * kMaxTopK + 4 * 2 * 4 * RBM +
                        sizeof(RouterParams);
    // the forward epilogue keeps the logits [n_pad][128] and the slice lists [4][KMAX][128] (values
    // and indices) in the idle ring
    if (!BWD && (size_t)a.p.stages * a.p.stage_bytes <
                    (size_t)a.p.n_pad * RBM * 4 + (size_t)4 * KMAX * RBM * 8)
        return cudaErrorInvalidValue;
    const int n_tiles = (m.T + RBM - 1) / RBM;
    const int threads = router_threads(BWD);
    auto kern = router_tc_kernel<KMAX, BWD>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    if (a.p.csize == 1) {
        e = launch_pdl(kern, dim3(n_tiles), dim3(threads), smem, st, a);
    } else {   // clusters of csize CTAs per tile
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(n_tiles * a.p.csize);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)a.p.csize;
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
    a.p.topk_idx = topk_idx;
    a.p.topk_gate = topk_gate;
    a.p.tile_counts = tile_counts;
    a.p.tile_psum = tile_psum;
    a.p.status = status;
    if (tables) {
        if (m.T > RBM) return cudaErrorInvalidValue;   // one tile only
        a.p.fused = 1;
        a.p.pad = tables->pad;
        a.p.counts_out = tables->counts;
        a.p.psum_out = tables->psum;
        a.p.offsets = tables->offsets;
        a.p.perm_token = tables->perm_token;
        a.p.perm_slot = tables->perm_slot;
        a.p.f_out = tables->f;
        a.p.P_out = tables->P;
        a.p.losses = tables->losses;
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
    a.p.topk_idx = const_cast<int*>(topk_idx);
    a.p.csize = 1;   // the backward epilogue needs the whole logit row of a token in one CTA
    a.p.dgate = dgate;
    a.p.counts = counts;
    a.p.dz = static_cast<__nv_bfloat16*>(dz);
    a.p.tile_dz = tile_dz;
    a.p.a1 = m.a1;
    a.p.a2 = m.a2;
    a.p.D = m.D;
    a.p.status = status;
    return launch_router_kernel<8, true>(m, a, st);
}

}  // namespace moe
