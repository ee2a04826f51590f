// permute_static.cu -- moe_permute_noalloc: the token -> expert grouping for
// callers that must not allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not allowed or not
// possible -- inside another framework's memory arena that forbids foreign
// allocations, in a real-time or embedded serving loop that freezes its
// device memory after start-up, or in an engine that only wants the grouping
// (to drive its own expert GEMMs) and has no use for a whole moe_layer with
// its multi-gigabyte weight copies.  moe_permute needs a layer, and making a
// layer allocates.  This entry point needs none: the counting sort's
// bookkeeping (per-expert counts, padded segment starts, tile scans, the
// padded row maps) lives in one file-scope __device__ array of fixed size
// that every GPU loading the library keeps until the process exits.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "layer.h"

namespace moe {

constexpr int kNoallocMaxRows = 65536;  // T * top_k per call
constexpr int kNoallocMaxPadded = kNoallocMaxRows + kMaxExperts * (kRowTile - 1);
// counts [E] + poff, tile_scan, chunk_scan [E+1] + row_pos [rows] + pos_row [padded rows]
constexpr size_t kNoallocWords = (size_t)kMaxExperts + 3 * (kMaxExperts + 1) + kNoallocMaxRows +
                                 kNoallocMaxPadded;

// 1,060,876 bytes on every device that loads the library.  In host code the
// name is only a handle; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocWords];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {};


// Once per device, with that device current: look up the array's device
// address and set the sort kernel's shared-memory limit.
cudaError_t setup(int dev, int32_t** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        e = kernels_init();
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const int32_t* ids, int T, int top_k, int n_experts,
                                          int32_t* offsets, int32_t* row_src, int32_t* row_dst,
                                          moe_stream_t stream) {
    using namespace moe;
    auto fail = [](moe_status st, const char* msg) {
        char buf[200];
        snprintf(buf, sizeof(buf), "moe_permute_noalloc: %s", msg);
        set_thread_error(buf);  // what moe_last_error(NULL) reports
        return st;
    };
    if (!ids || !offsets || !row_src || !row_dst) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    if (top_k < 1 || top_k > kMaxTopK) return fail(MOE_ERR_INVALID_ARG, "top_k must be in [1, 8]");
    if (n_experts < 1 || n_experts > kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "n_experts must be in [1, 1024]");
    if (T < 1 || (long long)T * top_k > kNoallocMaxRows)
        return fail(MOE_ERR_INVALID_ARG, "T * top_k must be in [1, 65536] (the static scratch size)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device ordinal above 63");
    int32_t* scratch = nullptr;
    e = setup(dev, &scratch);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    // The sort writes every scratch word it later reads within the same call
    // (counts and scans for e <= E, row_pos for every row, pos_row over the
    // padded range), so nothing has to be cleared between calls.
    int32_t* counts = scratch;
    int32_t* poff = counts + kMaxExperts;
    int32_t* tile_scan = poff + (kMaxExperts + 1);
    int32_t* chunk_scan = tile_scan + (kMaxExperts + 1);
    int32_t* row_pos = chunk_scan + (kMaxExperts + 1);
    int32_t* pos_row = row_pos + kNoallocMaxRows;
    e = launch_permute_raw(ids, T, top_k, n_experts, offsets, row_src, row_dst, counts, poff,
                           tile_scan, chunk_scan, row_pos, pos_row, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    return MOE_OK;
}
