// gemm_wgrad.cu -- weight-gradient GEMMs of the layer backward on tcgen05: C = A^T B, summed over
// the rows of each group, with A [rows, M] and B [rows, N] row-major bf16 (both operands
// MN-major for the MMA) and fp32 C written into the caller's gradient layouts.
//
// Weight gradients of the expert FFNs (chain rule through the FFN of [P1] "DeepSeekMoE 论文解读"
// (xxmr.cn), §方法细节): dW_down,e = sum_rows dy (x) act, dW_{gate|up},e = sum_rows d(gate|up) (x) x,
// and of the centroids: de_j = sum_t dz_{t,j} u_t.
//
// Group 0 is dense over T rows (the shared experts side by side, or the router's centroid
// gradient); routed group j reduces over its padded segment poff[j] .. poff[j+1]-1, whose rows
// past the expert's count are zero. Each K step is 64 rows: TMA brings A as two and B as four
// [64 rows x 64 columns] boxes with 128-byte swizzle, i.e. MN-major swizzle atoms of 8 rows x 128
// bytes; the MMA descriptors step through 16-row K slices (2 atoms) and across the 64-column boxes
// with the leading-byte offset. Same warp roles, TMEM double buffering and bounded waits as
// gemm_tc.cu.
//
// Tiles are claimed dynamically: the dense group's tiles reduce over all T rows and run an order
// of magnitude longer than a routed expert's, so a static round-robin leaves some SMs one long
// tile behind. The producer takes the next tile index from a global counter (zeroed by the
// caller before the launch; one claim ahead of the tile it loads) and hands each index to the MMA
// and epilogue warps through a small shared-memory ring; an index >= the tile count ends all roles.
//
// The fp32 results leave through TMA bulk stores: each epilogue warp stages its 32 rows x 16
// columns (a 2 KB box, 64-byte swizzle, so the thread-per-row writes are free of bank conflicts)
// in one of two shared buffers and one lane stores the box through a 3D tensor map
// [experts][rows][columns] of the output, whose extents clip rows and columns outside an expert.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "waits.cuh"

namespace moe {

namespace {

constexpr int WBM = 128, WBN = 256, WBK = 64, WSTAGES = 4, kWThreads = 192;
constexpr uint32_t kABytes = WBM * WBK * 2, kBBytes = WBN * WBK * 2, kBox = 64 * 64 * 2;
constexpr int kTileRing = 8;   // tile indices in flight between the producer and the consumers
constexpr uint32_t kStageBytes = 2 * 2 * 32 * 16 * 4;   // per epilogue warp: 2 buffers x 2 halves
constexpr size_t kWgradSmem = 1024 + (size_t)WSTAGES * (kABytes + kBBytes) + 4 * kStageBytes +
                              8 * (2 * WSTAGES + 5 + 2 * kTileRing) + 16 + 4 * kTileRing +
                              4 * (kMaxRouted + 2);
static_assert(kWgradSmem <= 232448, "shared memory of the weight-gradient kernel");

struct WgArgs {
    CUtensorMap a_r, a_s, b_r, b_s;   // [rows, M] / [rows, N], box [64 rows x 64 columns]
    const int* poff;                  // [n_routed + 1] padded segment starts
    int n_routed, has_shared, T;
    int M_r, N_r, M_s, N_s;           // C extents per group kind
    int mt_r, nt_r, mt_s, nt_s;       // tiles per group
    int mode;                         // 0: dW_down, 1: dW_gate / dW_up, 2: dense rows
    CUtensorMap out_map0, out_map1;   // fp32 outputs as [experts][rows][columns], 16-column boxes
    int Ks, I, d, n_valid_rows;
    int* tile_counter;                // zero at launch
    int* status;
};

struct WTile {
    int group, m_blk, n_blk, k_blocks, row0;
};

__device__ __forceinline__ WTile decode(int t, const WgArgs& a, const int* poff_s) {
    WTile w;
    const int tiles_s = a.has_shared ? a.mt_s * a.nt_s : 0;
    int local;
    if (t < tiles_s) {
        w.group = 0;
        local = t;
        w.m_blk = local / a.nt_s;
        w.n_blk = local % a.nt_s;
        w.k_blocks = (a.T + WBK - 1) / WBK;
        w.row0 = 0;
    } else {
        const int per = a.mt_r * a.nt_r;
        const int j = (t - tiles_s) / per;
        local = (t - tiles_s) % per;
        w.group = 1 + j;
        w.m_blk = local / a.nt_r;
        w.n_blk = local % a.nt_r;
        w.row0 = poff_s[j];
        w.k_blocks = (poff_s[j + 1] - poff_s[j]) / WBK;
    }
    return w;
}

// 128-byte-swizzled MN-major operand: atoms of 8 rows (K) x 128 bytes (64 MN elements); the
// stride-byte offset steps 8 K rows (1024 bytes), the leading-byte offset steps 64 MN elements.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo) {
    uint64_t desc = 0;
    desc |= (uint64_t)((saddr >> 4) & 0x3FFF);
    desc |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    desc |= (uint64_t)(1024 >> 4) << 32;
    desc |= (uint64_t)1 << 46;
    desc |= (uint64_t)2 << 61;
    return desc;
}

__global__ void __launch_bounds__(kWThreads, 1) wgrad_kernel(const __grid_constant__ WgArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_ring = base;
    uint8_t* b_ring = base + WSTAGES * kABytes;
    uint8_t* staging = base + WSTAGES * (kABytes + kBBytes);   // [4 warps][kStageBytes]
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + 4 * kStageBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + WSTAGES;
    uint64_t* tfull = bars + 2 * WSTAGES;
    uint64_t* tempty = bars + 2 * WSTAGES + 2;
    uint64_t* drain = bars + 2 * WSTAGES + 4;
    uint64_t* tile_full = drain + 1;             // [kTileRing]: an index was published
    uint64_t* tile_empty = tile_full + kTileRing; // [kTileRing]: MMA + 4 epilogue warps read it
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tile_empty + kTileRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* tile_idx = reinterpret_cast<volatile int*>(tmem_holder + 4);   // [kTileRing]
    int* poff_s = reinterpret_cast<int*>(tmem_holder + 4 + kTileRing);          // [n_routed + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < WSTAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_addr(&tfull[b]), 1);
            ptx::mbar_init(ptx::smem_addr(&tempty[b]), 4);
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        for (int r = 0; r < kTileRing; ++r) {
            ptx::mbar_init(ptx::smem_addr(&tile_full[r]), 1);
            ptx::mbar_init(ptx::smem_addr(&tile_empty[r]), 5);
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&a.a_r);
        ptx::prefetch_tmap(&a.a_s);
        ptx::prefetch_tmap(&a.b_r);
        ptx::prefetch_tmap(&a.b_s);
        ptx::prefetch_tmap(&a.out_map0);
        if (a.mode == 1) ptx::prefetch_tmap(&a.out_map1);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), 2 * WBN);
        ptx::tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    for (int j = threadIdx.x; j <= a.n_routed; j += blockDim.x) poff_s[j] = a.poff ? a.poff[j] : 0;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int total = (a.has_shared ? a.mt_s * a.nt_s : 0) + a.n_routed * a.mt_r * a.nt_r;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------------- TMA producer
            int stage = 0, issued = 0, slot = 0;
            uint32_t phase = 0, slot_phase = 0;
            bool ok = true;
            int next_t = atomicAdd(a.tile_counter, 1);
            while (ok) {
                const int t = next_t;
                if (!wait_phase(ptx::smem_addr(&tile_empty[slot]), slot_phase ^ 1, abort_flag,
                                a.status)) {
                    ok = false;
                    break;
                }
                tile_idx[slot] = t;
                ptx::mbar_arrive(ptx::smem_addr(&tile_full[slot]));
                if (++slot == kTileRing) {
                    slot = 0;
                    slot_phase ^= 1;
                }
                if (t >= total) break;
                next_t = atomicAdd(a.tile_counter, 1);
                const WTile w = decode(t, a, poff_s);
                const bool sh = w.group == 0;
                const CUtensorMap* am = sh ? &a.a_s : &a.a_r;
                const CUtensorMap* bm = sh ? &a.b_s : &a.b_r;
                for (int kb = 0; kb < w.k_blocks; ++kb) {
                    if (!wait_phase(ptx::smem_addr(&empty[stage]), phase ^ 1, abort_flag,
                                    a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::smem_addr(&full[stage]);
                    ptx::mbar_arrive_expect_tx(fb, kABytes + kBBytes);
                    const int y = w.row0 + kb * WBK;
                    const uint32_t as = ptx::smem_addr(a_ring + stage * kABytes);
                    const uint32_t bs = ptx::smem_addr(b_ring + stage * kBBytes);
#pragma unroll
                    for (int c = 0; c < WBM / 64; ++c)
                        ptx::tma_load_2d(as + c * kBox, am, w.m_blk * WBM + 64 * c, y, fb);
#pragma unroll
                    for (int c = 0; c < WBN / 64; ++c)
                        ptx::tma_load_2d(bs + c * kBox, bm, w.n_blk * WBN + 64 * c, y, fb);
                    ++issued;
                    if (++stage == WSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                for (int i = 0; i < issued && i < WSTAGES; ++i) {
                    if (--stage < 0) {
                        stage = WSTAGES - 1;
                        phase ^= 1;
                    }
                    drain_wait(ptx::smem_addr(&full[stage]), phase);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // -------------------------------------------------- MMA issuer
            const uint32_t idesc = ptx::idesc_bf16_f32(WBM, WBN) | (1u << 15) | (1u << 16);
            int stage = 0, acc = 0, slot = 0;
            uint32_t phase = 0, acc_phase = 0, slot_phase = 0;
            bool ok = true, any = false;
            while (ok) {
                if (!wait_phase(ptx::smem_addr(&tile_full[slot]), slot_phase, abort_flag, a.status))
                    break;
                const int t = tile_idx[slot];
                ptx::mbar_arrive(ptx::smem_addr(&tile_empty[slot]));
                if (++slot == kTileRing) {
                    slot = 0;
                    slot_phase ^= 1;
                }
                if (t >= total) break;
                const WTile w = decode(t, a, poff_s);
                if (!wait_phase(ptx::smem_addr(&tempty[acc]), acc_phase ^ 1, abort_flag,
                                a.status))
                    break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + acc * WBN;
                for (int kb = 0; kb < w.k_blocks; ++kb) {
                    if (!wait_phase(ptx::smem_addr(&full[stage]), phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_addr(a_ring + stage * kABytes);
                    const uint32_t b0 = ptx::smem_addr(b_ring + stage * kBBytes);
#pragma unroll
                    for (int k = 0; k < WBK / 16; ++k)   // 16 K rows = two swizzle atoms
                        ptx::mma_f16(d_tmem, sw128_mn_desc(a0 + k * 2048, kBox),
                                     sw128_mn_desc(b0 + k * 2048, kBox), idesc,
                                     (kb | k) != 0 ? 1u : 0u);
                    any = true;
                    ptx::mma_commit(ptx::smem_addr(&empty[stage]));
                    if (++stage == WSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_addr(&tfull[acc]));   // also when no K blocks ran
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (*abort_flag && any) {
                ptx::mma_commit(ptx::smem_addr(drain));
                drain_wait(ptx::smem_addr(drain), 0);
            }
        }
    } else {               // ---------------------------------------------------- epilogue
        const int quarter = warp & 3;
        uint8_t* my_stage = staging + (warp - 2) * kStageBytes;
        int acc = 0, slot = 0, sbuf = 0;
        uint32_t acc_phase = 0, slot_phase = 0;
        while (true) {
            int t = total;
            if (lane == 0) {
                if (wait_phase(ptx::smem_addr(&tile_full[slot]), slot_phase, abort_flag, a.status)) {
                    t = tile_idx[slot];
                    ptx::mbar_arrive(ptx::smem_addr(&tile_empty[slot]));
                }
            }
            t = __shfl_sync(0xffffffffu, t, 0);
            if (++slot == kTileRing) {
                slot = 0;
                slot_phase ^= 1;
            }
            if (t >= total) break;
            const WTile w = decode(t, a, poff_s);
            int ok = 1;
            if (lane == 0)
                ok = wait_phase(ptx::smem_addr(&tfull[acc]), acc_phase, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ptx::tc_fence_after();
            const bool sh = w.group == 0;
            const int M = sh ? a.M_s : a.M_r, Ncols = sh ? a.N_s : a.N_r;
            const int m0 = w.m_blk * WBM + quarter * 32;        // first C row of this warp
            const uint32_t t_base = tmem + acc * WBN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < WBN / 32; ++c) {
                const int col0 = w.n_blk * WBN + c * 32;
                if (col0 >= Ncols) break;
                uint32_t v[32];
                if (w.k_blocks > 0) {
                    ptx::tmem_ld_32x32b_x32(t_base + c * 32, v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;   // an expert without tokens
                }
                if (m0 >= M) continue;   // warp-uniform: rows past the C extent
                // the buffer written two chunks ago must have been read by its stores
                if (lane == 0) ptx::bulk_wait_read<1>();
                __syncwarp();
                uint8_t* buf = my_stage + sbuf * (kStageBytes / 2);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int pos = h * 2048 + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4);
                        *reinterpret_cast<uint4*>(buf + pos) =
                            make_uint4(v[16 * h + 4 * q], v[16 * h + 4 * q + 1],
                                       v[16 * h + 4 * q + 2], v[16 * h + 4 * q + 3]);
                    }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t sb = ptx::smem_addr(buf);
                    for (int h = 0; h < 2; ++h) {
                        const int cc = col0 + 16 * h;   // first C column of the box
                        if (cc >= Ncols) break;
                        if (a.mode == 1) {   // packed rows m0.. -> 16 gate rows, 16 up rows
                            const int ig = 16 * (m0 / 32);
                            const int e = sh ? ig / a.I : a.Ks + w.group - 1;
                            const int i = sh ? ig % a.I : ig;
                            ptx::tma_store_3d(&a.out_map0, sb + h * 2048, cc, i, e);
                            ptx::tma_store_3d(&a.out_map1, sb + h * 2048 + 1024, cc, i, e);
                        } else if (a.mode == 0) {   // C rows = model columns, C columns = i
                            const int e = sh ? cc / a.I : a.Ks + w.group - 1;
                            const int i = sh ? cc % a.I : cc;
                            ptx::tma_store_3d(&a.out_map0, sb + h * 2048, i, m0, e);
                        } else if (m0 < a.n_valid_rows) {   // dense: rows past N' are padding
                            ptx::tma_store_3d(&a.out_map0, sb + h * 2048, cc, m0, 0);
                        }
                    }
                    ptx::bulk_commit();
                }
                sbuf ^= 1;
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&tempty[acc]));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (lane == 0) ptx::bulk_wait_all();   // the stores read shared memory until they finish
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 2 * WBN);
    }
}

// [rows, cols] bf16 row-major as an MN-major operand: box of 64 rows x 64 columns.
bool encode_mn_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols) {
    return encode_bf16_map(map, ptr, rows, cols, 64);
}

// fp32 [experts, rows, cols] row-major output with a [1 x box_rows x 16] box, 64-byte swizzle.
bool encode_out_map(CUtensorMap* map, float* ptr, uint64_t experts, uint64_t rows, uint64_t cols,
                    int box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn || !ptr || experts == 0 || rows == 0 || cols == 0) return false;
    cuuint64_t dims[3] = {cols, rows, experts};
    cuuint64_t strides[2] = {cols * 4, rows * cols * 4};
    cuuint32_t box[3] = {16u, (cuuint32_t)box_rows, 1u};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_wgrad(const WgradSpec& s, int* status, cudaStream_t st) {
    WgArgs a{};
    if (s.n_routed > 0 && (!encode_mn_map(&a.a_r, s.a_r, s.rows_r, s.M_r) ||
                           !encode_mn_map(&a.b_r, s.b_r, s.rows_r, s.N_r)))
        return cudaErrorInvalidValue;
    if (s.has_shared && (!encode_mn_map(&a.a_s, s.a_s, s.T, s.M_s) ||
                         !encode_mn_map(&a.b_s, s.b_s, s.T, s.N_s)))
        return cudaErrorInvalidValue;
    if (s.n_routed == 0) {
        a.a_r = a.a_s;
        a.b_r = a.b_s;
    } else if (!s.has_shared) {
        a.a_s = a.a_r;
        a.b_s = a.b_r;
    }
    a.poff = s.poff;
    a.n_routed = s.n_routed;
    a.has_shared = s.has_shared;
    a.T = s.T;
    a.M_r = s.M_r;
    a.N_r = s.N_r;
    a.M_s = s.M_s;
    a.N_s = s.N_s;
    a.mt_r = (s.M_r + WBM - 1) / WBM;
    a.nt_r = (s.N_r + WBN - 1) / WBN;
    a.mt_s = (s.M_s + WBM - 1) / WBM;
    a.nt_s = (s.N_s + WBN - 1) / WBN;
    a.mode = s.mode;
    const uint64_t E = (uint64_t)s.Ks + s.n_routed;
    bool maps_ok;
    if (s.mode == 0)
        maps_ok = encode_out_map(&a.out_map0, s.out0, E, s.d, s.I, 32);
    else if (s.mode == 1)
        maps_ok = encode_out_map(&a.out_map0, s.out0, E, s.I, s.d, 16) &&
                  encode_out_map(&a.out_map1, s.out1, E, s.I, s.d, 16);
    else
        maps_ok = encode_out_map(&a.out_map0, s.out0, 1, s.n_valid_rows, s.N_s, 32);
    if (!maps_ok) return cudaErrorInvalidValue;
    a.Ks = s.Ks;
    a.I = s.I;
    a.d = s.d;
    a.n_valid_rows = s.n_valid_rows;
    a.tile_counter = s.tile_counter;
    a.status = status;
    const long total = (long)(s.has_shared ? a.mt_s * a.nt_s : 0) + (long)s.n_routed * a.mt_r * a.nt_r;
    if (total == 0) return cudaSuccess;
    if (!s.tile_counter) return cudaErrorInvalidValue;
    const size_t smem = kWgradSmem;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(wgrad_kernel), smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<long>(total, sm_count());
    e = launch_pdl(wgrad_kernel, dim3(grid), dim3(kWThreads), smem, st, a);
    note_launches(1);
    return e;
}

}  // namespace moe
