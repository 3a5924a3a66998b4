// permute_static.cu -- moe_permute_static: the dispatch permutation with its scratch held in a
// fixed device array of this library instead of a caller workspace.
//
// Some callers cannot hand the library a workspace: code that runs where device allocation is
// not allowed or not possible (an engine that reserves all device memory up front and forbids
// further cudaMalloc, a plugin that receives only its input and output buffers, a real-time loop
// that must not take the implicit synchronisation of cudaMalloc/cudaFree). For them this entry
// point keeps the permutation's scratch -- the per-tile expert histograms and the per-tile bases
// -- in `g_permute_scratch`, a file-scope __device__ array that every GPU which loads the library
// holds until the process exits. Nothing is allocated per call.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Two int32 tables of at most kStaticTileEntries entries each (tile histogram, tile bases).
constexpr size_t kStaticTileEntries = 131072;   // n_tiles * N' limit (512 KiB per table)
constexpr size_t kStaticScratchBytes = 2 * kStaticTileEntries * sizeof(int);

__device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

// Device address of g_permute_scratch for each device, looked up once with that device current.
// In host code the array's name is only a host-side stand-in, so kernels get this address. The
// cached address stays valid as long as the device's primary context does: a cudaDeviceReset
// while the library is loaded would leave it stale, so callers of moe_permute_static must not
// reset the device in between.
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

cudaError_t static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_permute_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_permute_static(const moe_config* cfg, const int32_t* topk_idx,
                                  const int32_t* counts, int32_t* offsets, int32_t* perm_token,
                                  int32_t* perm_slot, int32_t* status, moe_stream_t stream) {
    Dims m;
    const int rc = validate_config(cfg, &m);   // the rules of every other entry point
    if (rc != MOE_OK) return rc;
    if ((m.T > 0 && (!topk_idx || !perm_token || !perm_slot)) || !offsets)
        return MOE_ERR_INVALID_ARG;
    const size_t n_tiles = ((size_t)m.T + kRouteTile - 1) / kRouteTile;
    if (n_tiles * (size_t)m.N > kStaticTileEntries) return MOE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (static_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    int* tile_counts = static_cast<int*>(scratch);
    int* tile_base = tile_counts + kStaticTileEntries;
    cudaStream_t st = (cudaStream_t)stream;
    if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    // The kernels overwrite every table entry they later read, so nothing needs clearing.
    cudaError_t e = launch_tile_hist(m, topk_idx, tile_counts, status, st);
    if (e == cudaSuccess) {
        FinalizeArgs fa{};
        fa.m = m;
        fa.n_tiles = (int)n_tiles;
        fa.tile_counts = tile_counts;
        fa.counts_check = counts;
        fa.offsets = offsets;
        fa.tile_base = tile_base;
        fa.status = status;
        e = launch_route_finalize(fa, st);
    }
    if (e == cudaSuccess)
        e = launch_perm_scatter(m, topk_idx, offsets, tile_base, perm_token, perm_slot, st);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
