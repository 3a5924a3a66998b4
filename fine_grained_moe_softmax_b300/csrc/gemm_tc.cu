// gemm_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Expert FFN ([P1] "DeepSeekMoE 论文解读" (xxmr.cn), §方法细节, read as SwiGLU):
//   gate/up:  act = silu(A W_gate^T) * (A W_up^T)  (SwiGLU formed in the epilogue)
//   down:     y   = act W_down^T
// over one dense shared group (all T tokens; the K_s shared experts side by side) and N' routed
// groups (expert j: rows offsets[j] .. offsets[j+1]-1 of the permuted matrices).
//
// Kernel shape: persistent, one CTA per SM, 2 + EW warps.
//   warp 0      TMA producer: A tile [128 x 64] and B tile [BN x 64] (bf16, 128-byte swizzle) per
//               stage into a STAGES-deep shared-memory ring; BN = 256, 192, 160 or 128 columns,
//               the widest that pads the group widths by at most a tenth.
//   warp 1      allocates the TMEM of two BN-column accumulators (a power of two of columns); one
//               thread issues tcgen05.mma (M=128, N=BN, K=16) into one of them, and commits stage
//               releases and tile completion to mbarriers.
//   warps 2..   EW = 4 or 8 epilogue warps: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..; with 8 warps two share each lane quarter and split its columns),
//               then SwiGLU, SwiGLU backward or plain conversion to bf16. The plain and SwiGLU
//               epilogues stage each warp's 32 rows x 32 outputs (x 16 for SwiGLU) in shared memory
//               (swizzled) and write them with a TMA bulk store; the SwiGLU-backward epilogue, and
//               any warp whose rows cross the end of a group, store valid rows/columns directly.
// Two accumulators let the epilogue of tile i overlap the main loop of tile i+1. Every wait on an
// mbarrier is bounded in time; on expiry the kernel records MOE_ERR_TIMEOUT, stops issuing work,
// drains what it issued and frees its TMEM before returning.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "groups.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "waits.cuh"

namespace moe {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major bf16 matrix [rows, cols] as a 2D tensor map with a [box_rows x 64] box, 128-byte
// swizzle, zero fill outside the matrix.
bool encode_bf16_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                     int box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn || rows == 0 || cols == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Row-major bf16 matrix [rows, cols] as a 3D tensor map over (64-column chunk, row, chunk index)
// with a box of [chunks x box_rows x 64]: one copy lands `chunks` consecutive [box_rows x 64] tiles,
// each 128-byte swizzled exactly as a 2D box would be.
bool encode_bf16_map_chunks(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                            int box_rows, int chunks) {
    auto fn = tensor_map_encoder();
    if (!fn || rows == 0 || cols == 0 || cols % 64 != 0) return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, (cuuint32_t)chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Row-major bf16 output [rows, cols] with row stride ld (elements) as a 2D TMA map for stores,
// box [32 rows x box_cols columns] (32: 64-byte rows, 64-byte swizzle; 16: 32-byte rows, 32-byte
// swizzle); columns >= cols and rows >= rows are clipped.
static bool encode_out_map(CUtensorMap* map, void* ptr, uint64_t rows, uint64_t cols,
                           uint64_t ld, int box_cols = 32) {
    auto fn = tensor_map_encoder();
    if (!fn || !ptr || rows == 0 || cols == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, 32u};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_expert_gemms_simt(const Dims& m, const void* u, const void* x_perm,
                                     const void* packed, const int* offsets, void* act_r,
                                     void* act_s, void* y_r, void* y_s, cudaStream_t st,
                                     cudaEvent_t mid_event);

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                       // 64 bf16 = one 128-byte swizzle row

// Epilogue warps per EPI (below): 4 suffice for the forward epilogues; the SwiGLU-backward epilogue
// loads the saved gate/up values and does twice the arithmetic, and needs 8 to keep up.
constexpr int epi_warps(int epi) { return epi == 2 ? 8 : 4; }

struct TcArgs {
    CUtensorMap a_r, a_s, b_r, b_s;
    CUtensorMap o_r, o_s;         // EPI 0: outputs [rows, n_cols] with a [32 x 32] box
    const int* offsets;
    const int* counts;            // optional: rows per routed group (padded segments)
    GroupTiles gt;
    int k_blocks_r, k_blocks_s;
    int b_rows_per_expert;
    int n_cols_r, n_cols_s;       // valid GEMM columns per group
    __nv_bfloat16* out_r;
    __nv_bfloat16* out_s;
    int ld_r, ld_s;
    __nv_bfloat16* pre_r;         // optional (gate/up): raw accumulator values, packed columns,
    __nv_bfloat16* pre_s;         // unit-major (see pre_unit)
    int pre_rows_r, pre_rows_s;   // rows of the two buffers
    int* status;
    int preload;                  // see GroupedGemm::preload
};

// Output staging of the box-store epilogues: per epilogue warp two boxes of 32 rows x 32 bf16
// (EPI 0) or 32 rows x 16 bf16 (EPI 1: the SwiGLU of a 32-column chunk is 16 activations)
constexpr uint32_t out_box_bytes(int epi) { return epi == 0 ? 32 * 32 * 2 : 32 * 16 * 2; }
constexpr uint32_t staging_bytes(int epi) { return epi == 2 ? 0 : 4 * 2 * out_box_bytes(epi); }

// ABOX: rows of A loaded per tile. A batch of at most 64 tokens gives every group at most 64
// rows, so its A slot holds 64 rows (8 KB) and the ring gets one more stage; the MMA still reads
// 128 rows, the other 64 from the shared memory that follows (in bounds), and those rows' outputs
// are never stored (an output row depends only on its own A row).
// PAIR: the tile is computed by a CTA pair (below); each CTA holds its 128 rows of A and half of
// the tile's BN weight rows.
template <int BN, int STAGES, int EPI, int ABOX = BM, bool PAIR = false>
struct Smem {
    static_assert(ABOX == BM || ABOX == 64, "A rows per tile");
    static_assert(!PAIR || ABOX == BM, "pairs load whole 128-row A tiles");
    static constexpr uint32_t a_bytes = ABOX * BK * 2;
    static constexpr uint32_t b_bytes = (PAIR ? BN / 2 : BN) * BK * 2;
    static constexpr uint32_t ring = STAGES * (a_bytes + b_bytes);
    static constexpr uint32_t staging = staging_bytes(EPI);
    static constexpr uint32_t bars = 8 * (2 * STAGES + 5);
    static constexpr uint32_t tables = 4 * (3 * (kMaxRouted + 2));
    static constexpr uint32_t total = 1024 + ring + staging + bars + 16 + tables;
    static_assert(total <= 232448, "shared memory of the expert GEMM");
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// The saved raw gate/up values are stored unit-major: 16-byte unit u (packed columns 8u .. 8u+7)
// of row r at element (u * rows + r) * 8. A warp's 32 consecutive rows then write (gate/up
// epilogue) and read (SwiGLU-backward epilogue) 512 contiguous bytes per unit.
__device__ __forceinline__ size_t pre_unit(int unit, int rows, int row) {
    return ((size_t)unit * rows + row) * 8;
}

// The saved gate/up values of intermediate columns col0 .. col0+31 of one row (packed columns
// 2 col0 .. 2 col0 + 63, units col0/4 .. col0/4 + 7), of which the second half exists only when
// col0 + 16 < n_cols.
__device__ __forceinline__ void load_pre_chunk(uint4 (&buf)[8], const __nv_bfloat16* pre, int rows,
                                               int row, int col0, int n_cols, bool valid) {
    if (!valid || col0 >= n_cols) return;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        buf[q] = *reinterpret_cast<const uint4*>(pre + pre_unit(col0 / 4 + q, rows, row));
    if (col0 + 16 < n_cols) {
#pragma unroll
        for (int q = 4; q < 8; ++q)
            buf[q] = *reinterpret_cast<const uint4*>(pre + pre_unit(col0 / 4 + q, rows, row));
    }
}

// EPI: 0 plain bf16 store; 1 SwiGLU of packed gate/up column pairs (expert FFN forward);
// 2 SwiGLU backward: the accumulator is d_act, and with the saved gate/up values of the same rows
// (pre, packed) the epilogue writes d_gate / d_up (packed) to out.
//
// PAIR: the grid is made of clusters of two CTAs on neighbouring SMs, and each pair computes
// 256-row tiles with the CTA-pair form of the MMA. Each CTA loads its own 128 rows of A and half
// of the BN weight rows, so an SM reads 32 KB instead of 48 KB per 64-deep K block, and the ring
// has room for more stages. The even CTA issues the MMAs; both CTAs' loads count on its "full"
// barriers, its MMA completions arrive on both CTAs' "empty" and "tfull" barriers, and both CTAs'
// epilogue warps arrive on its "tempty" barriers. Each CTA's epilogue reads its own 128 rows of
// the accumulator from its own TMEM.
template <int BN, int STAGES, int EPI, int EW, int ABOX, bool PAIR>
__global__ void __launch_bounds__((2 + EW) * 32, 1)
    gemm_tc_kernel(const __grid_constant__ TcArgs args) {
    static_assert(EW == 4 || EW == 8, "4 or 8 epilogue warps");
    static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256 && (BN / 32) % (EW / 4) == 0,
                  "tile width: the MMA's N (a multiple of 16 up to 256), whole 32-column chunks");
    // two accumulators of BN columns; allocations are powers of two
    constexpr uint32_t kTmemCols = 2 * BN <= 256 ? 256u : 512u;
    static_assert(!PAIR || (EPI != 2 && BN % 32 == 0), "pair tiles: forward epilogues");
    constexpr int TM = PAIR ? 2 * BM : BM;   // rows of a tile
    using S = Smem<BN, STAGES, EPI, ABOX, PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_ring = base;
    uint8_t* b_ring = base + STAGES * S::a_bytes;
    uint8_t* staging = base + S::ring;   // [4 warps][2][out box] (EPI 0 and 1)
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + S::ring + S::staging);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = bars + 2 * STAGES + 2;
    uint64_t* drain = bars + 2 * STAGES + 4;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + S::ring + S::staging + S::bars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* prefix = reinterpret_cast<int*>(base + S::ring + S::staging + S::bars + 16);
    int* rows_s = prefix + (kMaxRouted + 2);
    int* row0_s = rows_s + (kMaxRouted + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const GroupTiles gt = args.gt;
    const uint32_t crank = PAIR ? ptx::cluster_ctarank() : 0;   // CTA of the pair
    const bool leader = crank == 0;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // this CTA's tile stream
    const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int row_off = (int)crank * BM;   // this CTA's rows inside a tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&tfull[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&tempty[a]), PAIR ? 2 * EW : EW);
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&args.a_r);
        ptx::prefetch_tmap(&args.a_s);
        ptx::prefetch_tmap(&args.b_r);
        ptx::prefetch_tmap(&args.b_s);
        if constexpr (EPI != 2) {
            ptx::prefetch_tmap(&args.o_r);
            ptx::prefetch_tmap(&args.o_s);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), kTmemCols);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(tmem_holder), kTmemCols);
            ptx::tmem_relinquish();
        }
    }
    // with preload, the tile tables are built before the wait for the preceding launch and the
    // producer thread waits on its own, after it has issued the first tile's weight loads
    const bool preload = !PAIR && args.preload != 0;
    const bool producer = warp == 0 && lane == 0;
    if (!preload) {
        pdl_wait();
        pdl_trigger();
    }
    build_tile_prefix<TM>(prefix, rows_s, row0_s, args.offsets, gt, args.counts,
                          args.status);   // syncs
    if (preload && !producer) {
        pdl_wait();
        pdl_trigger();
    }
    ptx::tc_fence_before();
    if constexpr (PAIR)
        ptx::cluster_sync();   // both CTAs' barriers are initialised before either uses the other's
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int total = prefix[gt.n_groups];
    const int s_tiles = prefix[1];   // the shared group's tiles come first in tile order
    const int s_start = shared_start(total, s_tiles, n_units, args.k_blocks_s > args.k_blocks_r);

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long issued = 0;
            bool ok = true;
            int pre = 0;   // K blocks of the first tile whose weights were loaded before the wait
            if (preload) {
                if (unit < total) {
                    const TileInfo ti = decode_tile<TM>(tile_at(unit, s_tiles, s_start), prefix,
                                                        rows_s, row0_s, gt);
                    const bool sh = ti.group == 0;
                    const int kb_n = sh ? args.k_blocks_s : args.k_blocks_r;
                    const int b_y = (sh ? 0 : (ti.group - 1) * args.b_rows_per_expert) +
                                    ti.n_blk * BN;
                    pre = kb_n < STAGES ? kb_n : STAGES;
                    // a fresh ring: stage kb is free; its barrier expects the A box as well
                    for (int kb = 0; kb < pre; ++kb) {
                        const uint32_t fb = ptx::smem_addr(&full[kb]);
                        ptx::mbar_arrive_expect_tx(fb, S::a_bytes + S::b_bytes);
                        ptx::tma_load_2d(ptx::smem_addr(b_ring + kb * S::b_bytes),
                                         sh ? &args.b_s : &args.b_r, kb * BK, b_y, fb);
                    }
                }
                pdl_wait();
                pdl_trigger();
            }
            for (int t = unit; t < total && ok; t += n_units) {
                const TileInfo ti =
                    decode_tile<TM>(tile_at(t, s_tiles, s_start), prefix, rows_s, row0_s, gt);
                const bool sh = ti.group == 0;
                const CUtensorMap* am = sh ? &args.a_s : &args.a_r;
                const CUtensorMap* bm = sh ? &args.b_s : &args.b_r;
                const int kb_n = sh ? args.k_blocks_s : args.k_blocks_r;
                const int a_y = ti.row0 + ti.m_blk * TM + row_off;
                const int b_y = (sh ? 0 : (ti.group - 1) * args.b_rows_per_expert) + ti.n_blk * BN +
                                (PAIR ? (int)crank * (BN / 2) : 0);
                for (int kb = 0; kb < kb_n; ++kb) {
                    if (t == unit && kb < pre) {   // the weights are in flight: the A box only
                        ptx::tma_load_2d(ptx::smem_addr(a_ring + stage * S::a_bytes), am, kb * BK,
                                         a_y, ptx::smem_addr(&full[stage]));
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                        continue;
                    }
                    if (!wait_phase<PAIR>(ptx::smem_addr(&empty[stage]), phase ^ 1, abort_flag,
                                          args.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::smem_addr(&full[stage]);
                    if constexpr (PAIR) {
                        // both CTAs' boxes count on the even CTA's barrier, which expects them all
                        if (leader) ptx::mbar_arrive_expect_tx(fb, 2 * (S::a_bytes + S::b_bytes));
                        const uint32_t cfb = leader ? fb : ptx::mapa(fb, 0);
                        ptx::tma_load_2d_pair(ptx::smem_addr(a_ring + stage * S::a_bytes), am,
                                              kb * BK, a_y, cfb);
                        ptx::tma_load_2d_pair(ptx::smem_addr(b_ring + stage * S::b_bytes), bm,
                                              kb * BK, b_y, cfb);
                    } else {
                        ptx::mbar_arrive_expect_tx(fb, S::a_bytes + S::b_bytes);
                        ptx::tma_load_2d(ptx::smem_addr(a_ring + stage * S::a_bytes), am, kb * BK,
                                         a_y, fb);
                        ptx::tma_load_2d(ptx::smem_addr(b_ring + stage * S::b_bytes), bm, kb * BK,
                                         b_y, fb);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (PAIR && ok) {
                // the even CTA's MMA completions arrive on this CTA's "empty" barriers: wait for
                // the last ones so that none arrives after the pair has exited
                int st2 = stage;
                uint32_t ph2 = phase;
                for (long i = 0; i < issued && i < STAGES; ++i) {
                    if (--st2 < 0) {
                        st2 = STAGES - 1;
                        ph2 ^= 1;
                    }
                    drain_wait<PAIR>(ptx::smem_addr(&empty[st2]), ph2);
                }
            }
            if (!ok) {
                // let the loads already issued land before the CTA can exit (the odd CTA of a
                // pair cannot observe its loads: it waits a fixed time before the exit instead)
                for (long i = 0; i < issued && i < STAGES && leader; ++i) {
                    if (--stage < 0) {
                        stage = STAGES - 1;
                        phase ^= 1;
                    }
                    drain_wait<PAIR>(ptx::smem_addr(&full[stage]), phase);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------- MMA issuer ----
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(TM, BN);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, any = false;
            for (int t = unit; t < total && ok; t += n_units) {
                const TileInfo ti =
                    decode_tile<TM>(tile_at(t, s_tiles, s_start), prefix, rows_s, row0_s, gt);
                const int kb_n = ti.group == 0 ? args.k_blocks_s : args.k_blocks_r;
                if (!wait_phase<PAIR>(ptx::smem_addr(&tempty[acc]), acc_phase ^ 1, abort_flag,
                                      args.status))
                    break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + acc * BN;
                for (int kb = 0; kb < kb_n; ++kb) {
                    if (!wait_phase<PAIR>(ptx::smem_addr(&full[stage]), phase, abort_flag,
                                          args.status)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_addr(a_ring + stage * S::a_bytes);
                    const uint32_t b0 = ptx::smem_addr(b_ring + stage * S::b_bytes);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = ptx::sw128_kmajor_desc(a0 + k * 32);
                        const uint64_t bd = ptx::sw128_kmajor_desc(b0 + k * 32);
                        if constexpr (PAIR)
                            ptx::mma_f16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                        else
                            ptx::mma_f16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    any = true;
                    if constexpr (PAIR)
                        ptx::mma_commit_pair(ptx::smem_addr(&empty[stage]), 3);
                    else
                        ptx::mma_commit(ptx::smem_addr(&empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    ptx::mma_commit_pair(ptx::smem_addr(&tfull[acc]), 3);
                else
                    ptx::mma_commit(ptx::smem_addr(&tfull[acc]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (*abort_flag && any) {   // make sure no MMA is still writing TMEM
                if constexpr (PAIR)
                    ptx::mma_commit_pair(ptx::smem_addr(drain), 1);
                else
                    ptx::mma_commit(ptx::smem_addr(drain));
                drain_wait<PAIR>(ptx::smem_addr(drain), 0);
            }
        }
    } else {
        // --------------------------------------------------------------------- epilogue ----
        constexpr int kChunks = BN / 32 / (EW / 4);     // 32-column chunks per warp and tile
        const int quarter = warp & 3;
        const int c_first = ((warp - 2) >> 2) * kChunks;
        constexpr uint32_t kOutBox = out_box_bytes(EPI);
        uint8_t* my_stage = staging + (EPI != 2 ? (warp - 2) * 2 * kOutBox : 0);
        int sbuf = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = unit; t < total; t += n_units) {
            const TileInfo ti =
                decode_tile<TM>(tile_at(t, s_tiles, s_start), prefix, rows_s, row0_s, gt);
            const bool sh = ti.group == 0;
            const int wrow0 = ti.m_blk * TM + row_off + quarter * 32;   // the warp's first row
            const int r = wrow0 + lane;                                  // row inside the group
            const bool valid = r < ti.m_rows;
            __nv_bfloat16* out = sh ? args.out_s : args.out_r;
            const int ld = sh ? args.ld_s : args.ld_r;
            const int n_cols = sh ? args.n_cols_s : args.n_cols_r;
            const size_t orow = (size_t)(ti.row0 + r) * ld;
            const int col_base = ti.n_blk * BN + c_first * 32;
            // all 32 rows of this warp lie inside the group: the box store cannot reach rows of
            // the next group
            const bool box_store = EPI != 2 && wrow0 + 32 <= ti.m_rows;
            // EPI 2 reads the saved gate/up values of its rows one chunk ahead, the first chunk
            // before the accumulator is ready, so that their DRAM latency overlaps the main loop
            // and the previous chunk's arithmetic.
            uint4 pre_buf[2][8];
            const __nv_bfloat16* pre_in = sh ? args.pre_s : args.pre_r;
            const int pre_rows = sh ? args.pre_rows_s : args.pre_rows_r;
            if constexpr (EPI == 2)
                load_pre_chunk(pre_buf[0], pre_in, pre_rows, ti.row0 + r, col_base, n_cols, valid);
            int ok = 1;
            if (lane == 0)
                ok = wait_phase<PAIR>(ptx::smem_addr(&tfull[acc]), acc_phase, abort_flag,
                                      args.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t t_base =
                tmem + acc * BN + c_first * 32 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                const int col0 = col_base + c * 32;
                if (col0 >= n_cols) break;
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(t_base + c * 32, v);
                if constexpr (EPI == 2) {
                    if (c + 1 < kChunks)
                        load_pre_chunk(pre_buf[(c + 1) & 1], pre_in, pre_rows, ti.row0 + r,
                                       col0 + 32, n_cols, valid);
                }
                ptx::tmem_ld_wait();
                if (!valid) continue;
                if constexpr (EPI == 1) {
                    __nv_bfloat16* pre = sh ? args.pre_s : args.pre_r;
                    if (pre) {   // the raw gate/up values, kept for the backward
                        uint32_t p[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            p[q] = pack_bf16x2(__uint_as_float(v[2 * q]),
                                               __uint_as_float(v[2 * q + 1]));
#pragma unroll
                        for (int q = 0; q < 4; ++q)   // packed columns col0.. = units col0/8..
                            *reinterpret_cast<uint4*>(
                                pre + pre_unit(col0 / 8 + q, pre_rows, ti.row0 + r)) =
                                make_uint4(p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
                    }
                    uint32_t o[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float g0 = __uint_as_float(v[2 * q]), g1 = __uint_as_float(v[2 * q + 1]);
                        const float u0 = __uint_as_float(v[16 + 2 * q]);
                        const float u1 = __uint_as_float(v[16 + 2 * q + 1]);
                        o[q] = pack_bf16x2(silu_f32(g0) * u0, silu_f32(g1) * u1);
                    }
                    if (box_store) {   // 32 rows x 16 activations through shared memory
                        if (lane == 0) ptx::bulk_wait_read<1>();
                        __syncwarp();
                        uint8_t* buf = my_stage + sbuf * kOutBox;
                        // 32-byte rows, 32-byte swizzle: 16-byte half q of row r sits at
                        // position q ^ ((r >> 2) & 1)
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            *reinterpret_cast<uint4*>(buf + lane * 32 +
                                                      ((q ^ ((lane >> 2) & 1)) << 4)) =
                                make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(sh ? &args.o_s : &args.o_r, ptx::smem_addr(buf),
                                              col0 / 2, ti.row0 + wrow0);
                            ptx::bulk_commit();
                        }
                        sbuf ^= 1;
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(out + orow + col0 / 2);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                } else if constexpr (EPI == 2) {
                    // columns col0 .. col0+31 are intermediate indices i; their gate/up values
                    // are the packed blocks col0/16 and col0/16 + 1 (32 values each) of pre_buf
                    const int halves = col0 + 16 < n_cols ? 2 : 1;
                    const uint4* raw = pre_buf[c & 1];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < halves) {
                            const __nv_bfloat162* p2 =
                                reinterpret_cast<const __nv_bfloat162*>(raw + 4 * h);
                            uint32_t o[16];
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float2 g2 = __bfloat1622float2(p2[q]);       // gate
                                const float2 u2 = __bfloat1622float2(p2[8 + q]);   // up
                                const float da0 = __uint_as_float(v[16 * h + 2 * q]);
                                const float da1 = __uint_as_float(v[16 * h + 2 * q + 1]);
                                const float s0 = __fdividef(1.0f, 1.0f + __expf(-g2.x));
                                const float s1 = __fdividef(1.0f, 1.0f + __expf(-g2.y));
                                o[q] = pack_bf16x2(da0 * u2.x * s0 * (1.0f + g2.x * (1.0f - s0)),
                                                   da1 * u2.y * s1 * (1.0f + g2.y * (1.0f - s1)));
                                o[8 + q] = pack_bf16x2(da0 * g2.x * s0, da1 * g2.y * s1);
                            }
                            uint4* dst = reinterpret_cast<uint4*>(out + orow + 2 * col0 + 32 * h);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                        }
                    }
                } else {
                    uint32_t o[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        o[q] = pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                    if (box_store) {
                        // the buffer written two chunks ago must have been read by its store
                        if (lane == 0) ptx::bulk_wait_read<1>();
                        __syncwarp();
                        uint8_t* buf = my_stage + sbuf * kOutBox;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(buf + lane * 64 +
                                                      ((q ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {   // columns past n_cols are clipped by the map
                            ptx::tma_store_2d(sh ? &args.o_s : &args.o_r, ptx::smem_addr(buf), col0,
                                              ti.row0 + wrow0);
                            ptx::bulk_commit();
                        }
                        sbuf ^= 1;
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(out + orow + col0);
                        // widths are multiples of 16: the second half of a chunk may lie past the end
                        const int halves = col0 + 16 < n_cols ? 2 : 1;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q < 2 * halves)
                                dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !leader)
                    ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_addr(&tempty[acc]), 0));
                else
                    ptx::mbar_arrive(ptx::smem_addr(&tempty[acc]));
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if constexpr (EPI != 2) {   // the box stores read shared memory until they finish
            if (lane == 0) ptx::bulk_wait_all();
        }
    }

    ptx::tc_fence_before();
    __syncthreads();   // every role of this CTA has finished
    if constexpr (PAIR) {
        // after an abort, loads of the odd CTA that the even one never waited for may still be
        // landing in this CTA's shared memory: give them time before the pair can exit
        if (*abort_flag && !leader) {
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 1000000ull) {
            }
        }
        __syncwarp();
        ptx::cluster_sync();   // neither CTA leaves while the other may still signal it
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem, kTmemCols);
        else
            ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------- host side ----

template <int BN, int STAGES, int EPI, int ABOX = BM>
cudaError_t launch_tc(const TcArgs& args, int max_tiles, cudaStream_t st) {
    using S = Smem<BN, STAGES, EPI, ABOX>;
    constexpr int EW = epi_warps(EPI);
    auto kern = gemm_tc_kernel<BN, STAGES, EPI, EW, ABOX, false>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), S::total);
    if (e != cudaSuccess) return e;
    const int grid = max(1, min(sm_count(), max_tiles));
    e = launch_pdl(kern, dim3(grid), dim3((2 + EW) * 32), S::total, st, args);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

// CTA-pair launch: clusters of two CTAs, as many clusters as fit on the GPU at once (at most one
// per 256-row tile), each pair looping over its share of the tiles; max_tiles counts pair tiles.
template <int BN, int STAGES, int EPI>
cudaError_t launch_tc_pair(const TcArgs& args, int max_tiles, cudaStream_t st) {
    using S = Smem<BN, STAGES, EPI, BM, true>;
    constexpr int EW = epi_warps(EPI);
    auto kern = gemm_tc_kernel<BN, STAGES, EPI, EW, BM, true>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), S::total);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * sm_count());
    cfg.blockDim = dim3((2 + EW) * 32);
    cfg.dynamicSmemBytes = S::total;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // clusters resident at once, per device (a persistent grid larger than that would leave the
    // last clusters waiting for the first ones to finish all their tiles)
    static int resident[64] = {0};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (resident[dev] == 0) {
        int n = 0;
        cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
        if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
        cfg.numAttrs = 2;
        if (n <= 0) return cudaErrorLaunchOutOfResources;
        resident[dev] = n;
    }
    cfg.gridDim = dim3(2 * std::max(1, std::min(resident[dev], max_tiles)));
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

// Tile width: the widest of 256 / 192 / 160 / 128 columns whose padding is at most a tenth of
// the computed columns, else the one with the least padding. Wider tiles read less operand data
// from L2 per FLOP; the 8-warp SwiGLU-backward epilogue needs a multiple of 64.
int pick_bn(int n_r, int n_s, int epi) {
    const int cands[4] = {256, 192, 160, 128};
    int best = 128;
    long best_pad = -1;
    for (int bn : cands) {
        if (epi == 2 && bn % 64 != 0) continue;
        long padded = 0, cols = 0;
        for (int n : {n_r, n_s}) {
            if (n <= 0) continue;
            cols += n;
            padded += (long)(n + bn - 1) / bn * bn;
        }
        if (cols == 0) return 256;
        if ((padded - cols) * 10 <= padded) return bn;
        if (best_pad < 0 || padded - cols < best_pad) {
            best = bn;
            best_pad = padded - cols;
        }
    }
    return best;
}

template <int EPI>
cudaError_t run_gemm(const GroupedGemm& g, int* status, cudaStream_t st) {
    const bool shared = g.has_shared;
    const int bn = pick_bn(g.n_routed > 0 ? g.n_cols_r : 0, shared ? g.n_cols_s : 0, EPI);
    // at most 64 tokens: every group (routed or shared) has at most 64 rows
    const bool small_a = EPI != 2 && bn == 256 && g.T_shared > 0 && g.T_shared <= 64;
    // 256-column tiles of the forward epilogues run as CTA pairs over 256-row tiles when the K
    // loop is long enough to amortise a pair tile's pipeline start (16+ blocks) and the launch
    // gains more from the lighter operand feed than it loses to rounding ragged groups up to 256
    // rows: launches with dense groups only, and the plain epilogue, whose 256-row tiles cost less
    // than the SwiGLU epilogue's (measured on the expert shapes of the pages' models).
    const int kb_min = std::min(g.n_routed > 0 ? (int)((g.k_r + BK - 1) / BK) : INT32_MAX,
                                shared ? (int)((g.k_s + BK - 1) / BK) : INT32_MAX);
    const bool pair = EPI != 2 && bn == 256 && !small_a && kb_min >= 16 &&
                      (EPI == 0 || g.n_routed == 0);
    const int a_box = small_a ? 64 : BM;
    const int b_box = pair ? bn / 2 : bn;
    TcArgs a{};
    if (g.n_routed > 0) {
        if (!encode_bf16_map(&a.a_r, g.a_r, g.a_rows_r, g.k_r, a_box) ||
            !encode_bf16_map(&a.b_r, g.b_r, g.b_rows_r, g.k_r, b_box))
            return cudaErrorInvalidValue;
    }
    if (shared) {
        if (!encode_bf16_map(&a.a_s, g.a_s, g.a_rows_s, g.k_s, a_box) ||
            !encode_bf16_map(&a.b_s, g.b_s, g.b_rows_s, g.k_s, b_box))
            return cudaErrorInvalidValue;
    }
    if (g.n_routed == 0) {   // a dense GEMM: only the shared slot has rows
        a.a_r = a.a_s;
        a.b_r = a.b_s;
    } else if (!shared) {    // the shared group is empty and never loads
        a.a_s = a.a_r;
        a.b_s = a.b_r;
    }
    a.offsets = g.offsets;
    a.counts = g.counts;
    a.gt.n_groups = 1 + g.n_routed;
    a.gt.has_shared = shared;
    a.gt.T = g.T_shared;
    a.gt.max_rows_r = (int)std::min<uint64_t>(g.a_rows_r, INT32_MAX);
    a.gt.n_tiles_r = (g.n_cols_r + bn - 1) / bn;
    a.gt.n_tiles_s = shared ? (g.n_cols_s + bn - 1) / bn : 0;
    // Shared-group weights above 64 MB do not stay in L2 while all row blocks pass over them:
    // panels of about 32 MB of weights each, so that A is read once per panel instead.
    const uint64_t b_col_bytes = (uint64_t)bn * g.k_s * 2;
    if (shared && (uint64_t)a.gt.n_tiles_s * b_col_bytes > (64ull << 20))
        a.gt.n_panel_s = (int)std::max<uint64_t>(1, (32ull << 20) / b_col_bytes);
    a.k_blocks_r = (int)((g.k_r + BK - 1) / BK);
    a.k_blocks_s = shared ? (int)((g.k_s + BK - 1) / BK) : 0;
    a.b_rows_per_expert = g.b_rows_per_expert;
    a.n_cols_r = g.n_cols_r;
    a.n_cols_s = g.n_cols_s;
    a.out_r = static_cast<__nv_bfloat16*>(g.out_r);
    a.out_s = static_cast<__nv_bfloat16*>(g.out_s);
    a.ld_r = g.ld_r;
    a.ld_s = g.ld_s;
    a.pre_r = static_cast<__nv_bfloat16*>(g.pre_r);
    a.pre_s = static_cast<__nv_bfloat16*>(g.pre_s);
    a.pre_rows_r = g.pre_rows_r;
    a.pre_rows_s = g.pre_rows_s;
    a.status = status;
    a.preload = g.preload;
    if (EPI != 2) {   // box-store maps of the outputs (the slot of an absent group copies the other)
        // EPI 1 writes one activation per gate/up column pair: half the GEMM's columns
        const int div = EPI == 1 ? 2 : 1, box_cols = EPI == 1 ? 16 : 32;
        const bool r_ok = g.n_routed > 0 &&
                          encode_out_map(&a.o_r, g.out_r, g.a_rows_r, (uint64_t)(g.n_cols_r / div),
                                         g.ld_r, box_cols);
        const bool s_ok = shared &&
                          encode_out_map(&a.o_s, g.out_s, g.T_shared, (uint64_t)(g.n_cols_s / div),
                                         g.ld_s, box_cols);
        if ((g.n_routed > 0 && !r_ok) || (shared && !s_ok)) return cudaErrorInvalidValue;
        if (!r_ok) a.o_r = a.o_s;
        if (!s_ok) a.o_s = a.o_r;
    }
    // upper bound of the tiles: sum over groups of ceil(M_j / 128) <= rows/128 + groups
    const long routed_mblk = g.n_routed > 0 ? (long)(g.max_routed_rows / BM) + g.n_routed : 0;
    const long max_tiles = routed_mblk * a.gt.n_tiles_r +
                           (long)((g.T_shared + BM - 1) / BM) * a.gt.n_tiles_s;
    const int mt = (int)std::min<long>(max_tiles, 1 << 30);
    if constexpr (EPI != 2) {
        if (pair) {   // tiles of 256 rows: sum over groups of ceil(M_j / 256)
            const long pr = g.n_routed > 0 ? (long)(g.max_routed_rows / (2 * BM)) + g.n_routed : 0;
            const long pt = pr * a.gt.n_tiles_r +
                            (long)((g.T_shared + 2 * BM - 1) / (2 * BM)) * a.gt.n_tiles_s;
            return launch_tc_pair<256, 6, EPI>(a, (int)std::min<long>(pt, 1 << 30), st);
        }
        if (small_a) return launch_tc<256, 5, EPI, 64>(a, mt, st);
    }
    if (bn == 256) return launch_tc<256, 4, EPI>(a, mt, st);
    if (bn == 192) return launch_tc<192, 5, EPI>(a, mt, st);
    if constexpr (EPI != 2) {
        if (bn == 160) return launch_tc<160, 5, EPI>(a, mt, st);
    }
    return launch_tc<128, 6, EPI>(a, mt, st);
}

}  // namespace

cudaError_t launch_expert_gemms(const Dims& m, const void* u, const void* x_perm,
                                const void* packed, const int* offsets, void* act_r, void* act_s,
                                void* y_r, void* y_s, int* status, cudaStream_t st,
                                cudaEvent_t mid_event, cudaEvent_t routed_ready,
                                cudaEvent_t main_start) {
    if (m.T == 0) {
        if (routed_ready) cudaStreamWaitEvent(st, routed_ready, 0);
        if (main_start) cudaEventRecord(main_start, st);
        if (mid_event) cudaEventRecord(mid_event, st);
        return cudaSuccess;
    }
    if (m.dtype == MOE_DTYPE_F32) {
        if (routed_ready) {
            const cudaError_t e = cudaStreamWaitEvent(st, routed_ready, 0);
            if (e != cudaSuccess) return e;
        }
        if (main_start) cudaEventRecord(main_start, st);
        return launch_expert_gemms_simt(m, u, x_perm, packed, offsets, act_r, act_s, y_r, y_s, st,
                                        mid_event);
    }
    const PackLayout P = pack_layout(m);
    const char* pk = static_cast<const char*>(packed);
    const uint64_t TK = (uint64_t)m.T * m.K, KsI = (uint64_t)m.Ks * m.I;
    GroupedGemm gu{};
    gu.n_routed = m.N;
    gu.has_shared = m.shared_active();
    gu.T_shared = m.T;
    gu.offsets = offsets;
    gu.max_routed_rows = (long)TK;
    // the offsets come from the router or the finalize kernel, ahead of the gather (or from the
    // caller), so both GEMMs may load their first weights while the preceding launch finishes.
    // Done for decode-sized batches, whose GEMMs stream weights and follow short launches (at
    // larger T no gain was measured)
    gu.preload = m.T <= 64 ? 1 : 0;
    gu.a_r = x_perm;
    gu.a_s = u;
    gu.b_r = pk + P.gu_r * 2;
    gu.b_s = pk + P.gu_s * 2;
    gu.a_rows_r = TK;
    gu.a_rows_s = m.T;
    gu.k_r = gu.k_s = m.d;
    gu.b_rows_r = (uint64_t)m.N * 2 * m.I;
    gu.b_rows_s = 2 * KsI;
    gu.b_rows_per_expert = 2 * m.I;
    gu.n_cols_r = 2 * m.I;
    gu.n_cols_s = (int)(2 * KsI);
    gu.out_r = act_r;
    gu.out_s = act_s;
    gu.ld_r = m.I;
    gu.ld_s = (int)KsI;
    cudaError_t e;
    if (routed_ready && gu.has_shared) {
        // the shared group needs only u: it runs first, while the routed rows are being gathered
        // on another stream; the routed groups follow once routed_ready has completed
        GroupedGemm gs = gu;
        gs.n_routed = 0;
        e = run_gemm<1>(gs, status, st);
        const cudaError_t ew = cudaStreamWaitEvent(st, routed_ready, 0);   // also after an error
        if (e == cudaSuccess) e = ew;
        GroupedGemm gr = gu;
        gr.has_shared = 0;
        if (main_start) cudaEventRecord(main_start, st);
        if (e == cudaSuccess) e = run_gemm<1>(gr, status, st);
    } else {
        if (routed_ready) e = cudaStreamWaitEvent(st, routed_ready, 0);
        else e = cudaSuccess;
        if (main_start) cudaEventRecord(main_start, st);
        if (e == cudaSuccess) e = run_gemm<1>(gu, status, st);
    }
    if (e != cudaSuccess) return e;
    if (mid_event) cudaEventRecord(mid_event, st);
    GroupedGemm dn = gu;
    dn.a_r = act_r;
    dn.a_s = act_s;
    dn.b_r = pk + P.dn_r * 2;
    dn.b_s = pk + P.dn_s * 2;
    dn.k_r = m.I;
    dn.k_s = KsI;
    dn.b_rows_r = (uint64_t)m.N * m.d;
    dn.b_rows_s = m.d;
    dn.b_rows_per_expert = m.d;
    dn.n_cols_r = dn.n_cols_s = m.d;
    dn.out_r = y_r;
    dn.out_s = y_s;
    dn.ld_r = dn.ld_s = m.d;
    return run_gemm<0>(dn, status, st);
}

cudaError_t run_grouped_gemm(const GroupedGemm& g, int epilogue, int* status, cudaStream_t st) {
    if (epilogue == 1) return run_gemm<1>(g, status, st);
    if (epilogue == 2) return run_gemm<2>(g, status, st);
    return run_gemm<0>(g, status, st);
}

}  // namespace moe
