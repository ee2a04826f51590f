// peaks.cu -- the denominators of the layer's rooflines, measured on the GPU
// the layer runs on: a plain HBM read stream (the decode and pp512 kernels
// are weight-read streams), a loop of block-scaled tcgen05 MMAs of the kind
// and shape the grouped GEMMs issue (kind::mxf8f6f4, M = 128, N = 256,
// K = 32, e4m3 A x e2m1 B, one UE8M0 scale per 32 elements), and the CUDA-core
// decode kernel's e2m1 dot-product rate (its arithmetic ceiling).
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

// ---- the CUDA-core decode kernel's arithmetic on one 32-block: 16 bytes of
// e2m1 codes -> f16 pairs by the hardware converter, times f16 operand values
// with fp32 accumulation (four partial sums of 8).
__device__ __forceinline__ void cvt_e2m1x8(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n.reg .b8 b0, b1, b2, b3;\nmov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\ncvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\ncvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
    asm("{\n.reg .b16 al, ah, bl, bh;\nmov.b32 {al, ah}, %1;\nmov.b32 {bl, bh}, %2;\n"
        "fma.rn.f32.f16 %0, al, bl, %0;\nfma.rn.f32.f16 %0, ah, bh, %0;\n}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}
__device__ __forceinline__ float dot_block(const uint4& w, const uint32_t (&op)[16]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h[4];
        cvt_e2m1x8(ws[i], h);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i] = fma2_f16_f32(h[j], op[4 * i + j], acc[i]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

constexpr int kDotWarps = 16;
constexpr int kDotSmem = 32768;

// 16 warps per CTA; each iteration a warp takes 4 distinct 512-byte chunks of
// a 32 KB shared-memory buffer (one 32-block per lane each, the chunks move
// every iteration and shared memory is declared clobbered, so no load or
// product carries over), as the decode kernel's compute warps do per stage.
// cyc[c]: clock cycles of CTA c's loop.
__global__ void __launch_bounds__(32 * kDotWarps, 1) k_dot_loop(const uint32_t* seed, int iters, float* out,
                                                               long long* cyc) {
    extern __shared__ __align__(16) uint8_t smd[];
    for (int i = threadIdx.x; i < kDotSmem / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(smd)[i] = seed[i & 1023];
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t op[16];
    for (int i = 0; i < 16; ++i) op[i] = seed[(lane * 16 + i) & 1023] & 0x3BFF3BFFu;  // finite f16 pairs
    float tot = 0.f;
    const long long c0 = clock64();
    for (int it = 0; it < iters; ++it) {
        asm volatile("" ::: "memory");
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int chunk = (warp * 4 + t + 4 * it) & 63;
            v[t] = dot_block(*reinterpret_cast<const uint4*>(smd + chunk * 512 + lane * 16), op);
        }
        tot += (v[0] + v[1]) + (v[2] + v[3]);
    }
    const long long c1 = clock64();
    out[blockIdx.x * blockDim.x + threadIdx.x] = tot;
    if (threadIdx.x == 0) cyc[blockIdx.x] = c1 - c0;
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

// `grid` CTAs of 16 warps each run `iters` iterations of 4 e2m1 32-block dot
// products per warp (4 x 1024 elements); seed: 1024 device words (the codes
// and operands), out: grid x 512 floats, cyc: grid int64 (each CTA's loop in
// clock cycles).  *ms = the kernel's duration.
int peak_dot_e2m1(int grid, int iters, const unsigned int* seed, float* out, long long* cyc, float* ms) {
    if (grid < 1 || iters < 1 || !seed || !out || !cyc || !ms) return (int)cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_dot_loop, cudaFuncAttributeMaxDynamicSharedMemorySize, kDotSmem);
    if (e != cudaSuccess) return (int)e;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return (int)cudaErrorUnknown;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return (int)cudaErrorUnknown;
    }
    cudaEventRecord(e0, 0);
    k_dot_loop<<<grid, 32 * kDotWarps, kDotSmem>>>(seed, iters, out, cyc);
    cudaEventRecord(e1, 0);
    int rc = (int)cudaDeviceSynchronize();
    if (rc == 0) rc = (int)cudaGetLastError();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

}  // extern "C"
