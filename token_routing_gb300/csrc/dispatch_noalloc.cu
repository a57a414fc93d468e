// moe_dispatch_noalloc: the dispatch step (capacity, counting sort into expert buckets,
// gather of x) for callers that cannot allocate device memory.
//
// Some callers have no way to allocate: code running where cudaMalloc is not allowed
// (inside a pre-allocated memory budget or a host framework that owns every allocation),
// or plugins that are handed only their input and output buffers. For them this entry
// point takes no workspace argument. Its sort scratch is a fixed array in the library's
// own device memory, reserved on every GPU that loads the library until the process
// exits. The arithmetic is that of moe_dispatch (same kernels, same results).
#include "internal.cuh"

namespace moe {

namespace {

// The library's own dispatch scratch. In host code this name is only a stand-in for the
// device symbol: host code must use the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_dispatch_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up on every call (a host
// lookup, no device work): after a device reset the module is loaded again and the array may
// sit elsewhere, so a cached address could point the sort at memory it does not own.
cudaError_t scratch_address(void** out) {
    return cudaGetSymbolAddress(out, g_dispatch_scratch);
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const int32_t* idx,
                                                     const void* x, int32_t* kept, int32_t* offsets,
                                                     int32_t* row_token, int32_t* slot_row,
                                                     int32_t* n_dropped, void* Xp, moe_stream_t stream) {
    const moe_status_t st = config_status(cfg);
    if (st != MOE_OK) return st;
    if (!kept || !offsets || !n_dropped) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!idx || !x || !slot_row)) return MOE_ERR_INVALID_ARG;
    if (cfg->rows_capacity > 0 && (!row_token || !Xp)) return MOE_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(Xp)) & 15u) != 0) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (dense_routing(*cfg)) {
        // closed-form layout: no scratch, no size limit
        if (launch_dense_layout(*cfg, idx, kept, offsets, row_token, slot_row, n_dropped, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (launch_gather(*cfg, x, offsets, row_token, slot_row, Xp, s) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (cfg->T > MOE_NOALLOC_MAX_TOKENS || (int64_t)cfg->T * cfg->k > MOE_NOALLOC_MAX_ASSIGNMENTS)
        return MOE_ERR_UNSUPPORTED;
    Workspace probe{nullptr, 0};
    SortScratch srt;
    sort_scratch_take(probe, *cfg, &srt);
    if (probe.used > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;

    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
    // Every scratch word the sort reads is written earlier in the same call, so the
    // previous call's leftovers need no clearing.
    Workspace ws{static_cast<char*>(base), 0};
    sort_scratch_take(ws, *cfg, &srt);
    if (launch_sort(*cfg, idx, srt, kept, offsets, row_token, slot_row, n_dropped, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_gather(*cfg, x, offsets, row_token, slot_row, Xp, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}
