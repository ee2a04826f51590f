// tc_probe.cu -- test-only single-tile checks of the tensor-core building
// blocks libmoe's tcgen05 kernels use (built and called by
// tests/test_gpu_tc_blocks.py; not part of the library).
//
//  probe_tma4: one 128x128 e2m1 tile loaded by TMA with the 16-byte-aligned
//    4-bit unpacking, on a barrier armed with the 8192 packed bytes the copy
//    delivers; reports that the barrier completed and dumps the shared-memory
//    image.
//  probe_mma: one M=128, N=32, K=128 block-scaled MMA (e2m1 x e4m3, UE8M0
//    scales per 32) through the same descriptors, scale-factor atoms and
//    tensor-memory copies as the library; returns D and the scale columns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "tc_ptx.cuh"

using namespace moe::tc;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

static EncodeTiledFn encode() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
}

static int make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows, bool fp4,
                    bool swizzle = true) {
    EncodeTiledFn enc = encode();
    if (!enc) return -1;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {fp4 ? cols / 2 : cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

constexpr uint64_t kLimit = 2000000ull;  // 2 ms

__global__ void k_probe_tma4(const __grid_constant__ CUtensorMap tm, uint8_t* dump, int* flags) {
    __shared__ __align__(1024) uint8_t buf[16384];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b0 = smem_u32(&bar);
    for (int i = threadIdx.x; i < 16384; i += blockDim.x) buf[i] = 0xEE;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(b0, 1);
        fence_mbar_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
        // a 128x128 e2m1 box counts its packed bytes: 128 rows x 64
        mbar_arrive_expect_tx(b0, 8192);
        tma_load_2d(smem_u32(buf), &tm, 0, 0, b0);
        const bool d0 = mbar_wait(b0, 0, kLimit, &abort_flag);
        if (!d0) spin_ns(200000);  // (not expected) let the copy land before the dump
        flags[0] = d0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 16384; i += blockDim.x) dump[i] = buf[i];
}

extern "C" int probe_tma4(const uint8_t* a_fp4, uint8_t* dump, int* flags) {
    CUtensorMap tm;
    int r = make_map(&tm, a_fp4, 128, 128, 128, true);
    if (r) return 1000 + r;
    k_probe_tma4<<<1, 128>>>(tm, dump, flags);
    return (int)cudaDeviceSynchronize();
}

__global__ void k_probe_mma(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const uint8_t* sfa, const uint8_t* sfb, int mode, uint32_t a_tx, uint32_t a_fmt,
                            float* d_out, uint32_t* sf_dump, int* flags) {
    __shared__ __align__(1024) uint8_t A[16384];
    __shared__ __align__(1024) uint8_t B[4096];
    __shared__ __align__(16) uint8_t SA[512];
    __shared__ __align__(16) uint8_t SB[512];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ uint32_t slot;
    __shared__ int abort_flag;
    __shared__ int ok_all;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t b0 = smem_u32(&bars[0]), b1 = smem_u32(&bars[1]);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ok_all = 0;
        mbar_init(b0, 1);
        mbar_init(b1, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&slot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(b0, a_tx + 4096 + 1024);
        tma_load_2d(smem_u32(A), &tmA, 0, 0, b0);
        tma_load_2d(smem_u32(B), &tmB, 0, 0, b0);
        bulk_load(smem_u32(SA), sfa, 512, b0);
        bulk_load(smem_u32(SB), sfb, 512, b0);
        const bool ok = mbar_wait(b0, 0, kLimit, &abort_flag);
        bool ok2 = false;
        if (ok) {
            tc_fence_after();
            tmem_cp_32x128_x4(tmem + 128, desc_sf(smem_u32(SA)));
            tmem_cp_32x128_x4(tmem + 132, desc_sf(smem_u32(SB)));
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t id = (mode == 0) ? kk : 0;
                const uint32_t off = (mode == 0) ? 0 : kk;
                mma_mx(tmem, desc_sw128(smem_u32(A) + 32 * kk), desc_sw128(smem_u32(B) + 32 * kk),
                       idesc_mx(a_fmt, kFmtE4M3, 128, 32, id, id), tmem + 128 + off, tmem + 132 + off,
                       kk > 0 ? 1u : 0u);
            }
            mma_commit(b1);
            ok2 = mbar_wait(b1, 0, kLimit, &abort_flag);
        }
        if (!ok || !ok2) spin_ns(200000);
        flags[0] = ok;
        flags[1] = ok2;
        ok_all = ok && ok2;
    }
    __syncthreads();
    tc_fence_after();
    if (ok_all) {
        const uint32_t tq = tmem + ((uint32_t)(32 * warp) << 16);
        uint32_t r0[16], r1[16], s0[16];
        tmem_ld16(tq, r0);
        tmem_ld16(tq + 16, r1);
        tmem_ld16(tq + 128, s0);
        tmem_ld_wait();
        const int m = 32 * warp + lane;
        for (int i = 0; i < 16; ++i) {
            d_out[m * 32 + i] = __uint_as_float(r0[i]);
            d_out[m * 32 + 16 + i] = __uint_as_float(r1[i]);
        }
        for (int i = 0; i < 8; ++i) sf_dump[m * 8 + i] = s0[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// a: [128][64] packed e2m1 (a_fmt 5) or [128][128] e4m3 (a_fmt 0); b: [32][128] e4m3;
// sfa, sfb: 512-byte atoms; d_out [128][32] f32; sf_dump [128][8] u32; flags [2].
extern "C" int probe_mma(const uint8_t* a, const uint8_t* b, const uint8_t* sfa, const uint8_t* sfb, int mode,
                         uint32_t a_tx, uint32_t a_fmt, float* d_out, uint32_t* sf_dump, int* flags) {
    CUtensorMap ta, tb;
    int r = make_map(&ta, a, 128, 128, 128, a_fmt == kFmtE2M1);
    if (r) return 1000 + r;
    r = make_map(&tb, b, 128, 32, 32, false);
    if (r) return 2000 + r;
    k_probe_mma<<<1, 128>>>(ta, tb, sfa, sfb, mode, a_tx, a_fmt, d_out, sf_dump, flags);
    return (int)cudaDeviceSynchronize();
}
