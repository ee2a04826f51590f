// peaks.cu -- the two denominators of the layer's rooflines, measured on the
// GPU the layer runs on: a plain HBM read stream (the decode and pp512
// kernels are weight-read streams) and a loop of block-scaled tcgen05 MMAs
// of the kind and shape the grouped GEMMs issue (kind::mxf8f6f4, M = 128,
// N = 256, K = 32, e4m3 A x e2m1 B, one UE8M0 scale per 32 elements).
// Built into its own library (libmoe_peaks.so); the layer never calls it.
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/moe_peaks.h"
#include "../csrc/tc_ptx.cuh"

using namespace moe::tc;

namespace {

// Every thread streams 16-byte loads (evict-first) over its grid stride and
// folds them into one word, so the loads cannot be dropped.
__global__ void k_read_stream(const uint4* __restrict__ p, long long n, unsigned int* sink) {
    unsigned int acc = 0;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint4 v = __ldcs(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x9E3779B9u) atomicAdd(sink, 1u);
}

constexpr int kABytes = 16384;  // 128 token rows x 128 bytes
constexpr int kBBytes = 32768;  // 256 weight rows x 128 bytes (e2m1 codes in 16-byte slots)
constexpr int kSmem = kABytes + kBBytes + 1024 + 64;
constexpr uint64_t kWaitNs = 2000000000ull;

// One thread per CTA issues `iters` groups of four K = 32 MMAs into one
// accumulator (columns 0-255) on operands resident in shared memory, then
// commits and waits (bounded) for the last group.  The issuing thread is
// throttled by the tensor pipe, so only the last few groups are in flight
// when it commits.  ok_out is cleared if the wait gave up.
__global__ void __launch_bounds__(64, 1) k_mma_loop(int iters, int* ok_out) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kABytes + kBBytes);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
    const int warp = threadIdx.x >> 5;
    // e4m3 0x38 = 1.0 in every A byte; the B bytes hold e2m1 1.0 pairs
    for (int i = threadIdx.x; i < (kABytes + kBBytes) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(sm)[i] = i < kABytes / 4 ? 0x38383838u : 0x22222222u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(sm), b = smem_u32(sm + kABytes);
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_mx(tmem, desc_sw128(a + 32 * kk), desc_sw128(b + 32 * kk),
                       idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk), tmem + 256, tmem + 260,
                       (it | kk) ? 1u : 0u);
        mma_commit(smem_u32(bar));
        if (!mbar_wait(smem_u32(bar), 0, kWaitNs, abort_flag)) {
            atomicExch(ok_out, 0);
            spin_ns(200000);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

extern "C" {

// Reads `bytes` (a multiple of 16) at p once with a grid of `grid` x 512
// threads; *ms = the kernel's duration (CUDA events on the legacy stream).
// Returns a cudaError_t code.
int peak_read_stream(const void* p, long long bytes, int grid, unsigned int* sink, float* ms) {
    if (!p || bytes < 16 || bytes % 16 || grid < 1 || !sink || !ms) return (int)cudaErrorInvalidValue;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return (int)cudaErrorUnknown;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return (int)cudaErrorUnknown;
    }
    cudaEventRecord(e0, 0);
    k_read_stream<<<grid, 512>>>(reinterpret_cast<const uint4*>(p), bytes / 16, sink);
    cudaEventRecord(e1, 0);
    int rc = (int)cudaDeviceSynchronize();
    if (rc == 0) rc = (int)cudaGetLastError();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// `grid` CTAs (one per SM) each issue iters x 4 block-scaled MMAs of
// 2 * 128 * 256 * 32 flops; *ms = the kernel's duration, *ok = 1 unless a
// CTA's final wait gave up.  Returns a cudaError_t code.
int peak_mma_mx(int grid, int iters, int* ok, float* ms) {
    if (grid < 1 || iters < 1 || !ok || !ms) return (int)cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_mma_loop, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return (int)e;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return (int)cudaErrorUnknown;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return (int)cudaErrorUnknown;
    }
    cudaEventRecord(e0, 0);
    k_mma_loop<<<grid, 64, kSmem>>>(iters, ok);
    cudaEventRecord(e1, 0);
    int rc = (int)cudaDeviceSynchronize();
    if (rc == 0) rc = (int)cudaGetLastError();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

}  // extern "C"
