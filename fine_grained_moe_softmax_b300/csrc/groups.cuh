// groups.cuh -- tile enumeration of the grouped expert GEMMs.
//
// Group 0 is the dense shared group (all T tokens, present when K_s > 0); groups 1..N' are the
// routed experts, expert j owning rows offsets[j] .. offsets[j+1]-1 of the permuted matrices.
// A group of M rows and Nc output columns has ceil(M/BM) * ceil(Nc/BN) tiles, enumerated with the
// column tile fastest so that CTAs running at the same time share the group's A rows and weights
// through L2. Tile t of the whole launch belongs to the group g with prefix[g] <= t < prefix[g+1].
// When the shared group's weights are too large to stay in L2 while every row block passes over
// them, its column tiles are cut into panels of n_panel_s columns, enumerated one after another
// (all row blocks of a panel, column fastest, before the next panel): the weights of a panel stay
// in L2 and A is read once per panel.
#pragma once

#include "common.cuh"

namespace moe {

struct GroupTiles {
    int n_groups;      // 1 + N'
    int has_shared;    // K_s > 0 (group 0 is empty otherwise)
    int T;             // rows of the shared group
    int n_tiles_r;     // column tiles of a routed group
    int n_tiles_s;     // column tiles of the shared group
    int max_rows_r;    // rows of the routed A / output matrices
    int n_panel_s;     // column tiles per panel of the shared group (<= 0: one panel)
};

struct TileInfo {
    int group;         // 0 = shared, 1 + j = routed expert j
    int m_rows;        // rows of the group
    int row0;          // first row of the group in its A / output matrix
    int m_blk, n_blk;  // tile coordinates inside the group
};

// Fills prefix[0 .. n_groups] (shared memory) from offsets; every thread of the CTA must call it.
// With `counts`, routed expert j has counts[j] rows starting at offsets[j] (padded segments);
// otherwise its rows are offsets[j] .. offsets[j+1]-1. A group reaching outside
// [0, gt.max_rows_r) (corrupt offsets from a caller) is cut to the rows inside and reported as
// MOE_ERR_CORRUPT_INPUT, so no tile can address rows outside the routed matrices.
template <int BM>
__device__ __forceinline__ void build_tile_prefix(int* prefix, int* rows_s, int* row0_s,
                                                  const int* __restrict__ offsets,
                                                  const GroupTiles& gt,
                                                  const int* __restrict__ counts = nullptr,
                                                  int* status = nullptr) {
    const int N = gt.n_groups - 1;
    for (int j = threadIdx.x; j <= N; j += blockDim.x) {
        if (j == 0) {
            rows_s[0] = gt.has_shared ? gt.T : 0;
            row0_s[0] = 0;
        } else {
            int lo = offsets[j - 1];
            int rows = counts ? counts[j - 1] : offsets[j] - lo;
            if (lo < 0 || lo > gt.max_rows_r || rows < 0 || rows > gt.max_rows_r - lo) {
                if (status) set_status(status, MOE_ERR_CORRUPT_INPUT);
                lo = min(max(lo, 0), gt.max_rows_r);
                rows = min(max(rows, 0), gt.max_rows_r - lo);
            }
            rows_s[j] = rows;
            row0_s[j] = lo;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        prefix[0] = 0;
        for (int g = 0; g <= N; ++g) {
            const int nt = g == 0 ? gt.n_tiles_s : gt.n_tiles_r;
            acc += ((rows_s[g] + BM - 1) / BM) * nt;
            prefix[g + 1] = acc;
        }
    }
    __syncthreads();
}

// Tile t of a persistent launch runs on unit t mod U (U = units of the grid), so with R = total
// mod U > 0 the units below R get one tile more. When the shared group's S tiles are longer than
// the routed ones (a longer K loop: the down GEMM, whose shared group is K_s experts deep) and few
// (S <= U - R and S <= total - R, as in a decode-sized batch), they are moved to positions
// R .. R+S-1, onto units with one tile less; the routed tiles keep their order around them.
// shared_start() gives R (0: positions are tile indices), tile_at() the tile of position p.
__device__ __forceinline__ int shared_start(int total, int s_tiles, int units, bool shared_longer) {
    if (!shared_longer || s_tiles <= 0 || units <= 0) return 0;
    const int rem = total % units;   // positions 0 .. R-1 need R routed tiles
    return (rem > 0 && rem + s_tiles <= units && rem + s_tiles <= total) ? rem : 0;
}
__device__ __forceinline__ int tile_at(int p, int s_tiles, int start) {
    if (start == 0) return p;
    if (p < start) return s_tiles + p;
    return p < start + s_tiles ? p - start : p;
}

template <int BM>
__device__ __forceinline__ TileInfo decode_tile(int t, const int* prefix, const int* rows_s,
                                                const int* row0_s, const GroupTiles& gt) {
    int lo = 0, hi = gt.n_groups - 1;   // find g with prefix[g] <= t < prefix[g+1]
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    TileInfo ti;
    ti.group = lo;
    ti.m_rows = rows_s[lo];
    ti.row0 = row0_s[lo];
    const int nt = lo == 0 ? gt.n_tiles_s : gt.n_tiles_r;
    const int local = t - prefix[lo];
    const int pw = lo == 0 && gt.n_panel_s > 0 && gt.n_panel_s < nt ? gt.n_panel_s : nt;
    if (pw == nt) {
        ti.m_blk = local / nt;
        ti.n_blk = local % nt;
    } else {
        const int mb = (ti.m_rows + BM - 1) / BM;
        const int full = nt / pw;                 // panels of pw columns, then one narrower
        const int per_panel = mb * pw;
        const int p = min(local / per_panel, full);
        const int w = p < full ? pw : nt - full * pw;
        const int r = local - p * per_panel;
        ti.m_blk = r / w;
        ti.n_blk = p * pw + r % w;
    }
    return ti;
}

}  // namespace moe
