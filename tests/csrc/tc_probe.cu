// tc_probe.cu -- test-only single-tile checks of the tensor-core building
// blocks libmoe's tcgen05 kernels use (built and called by
// tests/test_gpu_tc_blocks.py; not part of the library).
//
//  probe_tma4: one 128x128 e2m1 tile loaded by TMA with the 16-byte-aligned
//    4-bit unpacking; reports whether a barrier expecting 16384 transaction
//    bytes completes (waits are bounded) and dumps the shared-memory image.
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
    __shared__ __align__(1024) uint8_t buf0[16384];
    __shared__ __align__(1024) uint8_t buf1[16384];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;
    const uint32_t b0 = smem_u32(&bars[0]), b1 = smem_u32(&bars[1]);
    for (int i = threadIdx.x; i < 16384; i += blockDim.x) { buf0[i] = 0xEE; buf1[i] = 0xEE; }
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(b0, 1);
        mbar_init(b1, 1);
        fence_mbar_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(b0, 8192);
        tma_load_2d(smem_u32(buf0), &tm, 0, 0, b0);
        mbar_arrive_expect_tx(b1, 16384);
        tma_load_2d(smem_u32(buf1), &tm, 0, 0, b1);
        const bool d0 = mbar_wait(b0, 0, kLimit, &abort_flag);
        const bool d1 = mbar_wait(b1, 0, kLimit, &abort_flag);
        spin_ns(200000);
        flags[0] = d0;
        flags[1] = d1;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 16384; i += blockDim.x) dump[i] = buf1[i];
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

// ------------------------------------------------------------------------
// Microbenchmarks (timing only; results are not checked for values).
// ------------------------------------------------------------------------

// Block-scaled MMA with the A operand read from tensor memory (128 lanes x
// K/4 columns of 8-bit codes) instead of shared memory.
__device__ __forceinline__ void mma_mx_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], [%1], %2, %3, [%4], [%5], p;\n}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Streams `tiles_per_cta` x KB fp4 weight tiles (128 x 128) per CTA through a
// `stages`-deep TMA pipeline.  mode bit 0: issue one M=128,N=32 block-scaled
// MMA group per stage (else the consumer frees the stage at once); bit 1:
// prefetch tiles into L2 `pf` stages ahead.  CTA 0 records, per stage, the
// global time the load was issued and the time the consumer saw it land.
// kTA: the token operand of the swapped MMAs (mode bit 6) in tensor memory
// (its own instantiation: kernels holding that MMA form time differently)
template <bool kTA>
__global__ void __launch_bounds__(96, 1)
k_stream(const __grid_constant__ CUtensorMap tmA, int tiles_per_cta, int KB, int stages, int mode, int pf,
         unsigned long long* stamps, int* ok_out, int layout, uint32_t box_tx, uint32_t slot, const uint8_t* sf_src) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + stages * slot + 16384 + 1024);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * stages + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t b0 = smem_u32(bars);
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) { mbar_init(b0 + 8 * s, 1); mbar_init(b0 + 8 * (stages + s), 1); }
        mbar_init(b0 + 8 * (2 * stages), 1);
        mbar_init(b0 + 8 * (2 * stages + 1), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int total = tiles_per_cta * KB;
    bool ok = true;
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < total && ok; ++i) {
            const int s = i % stages;
            const uint32_t ph = (uint32_t)((i / stages) & 1);
            const int row = (blockIdx.x + (i / KB) * gridDim.x) * 128, kb = i % KB;
            if ((mode & 2) && i + pf < total) {
                // the tile the load of stage j will read (the coordinates of the branches below)
                const int j = i + pf;
                const int jrow = (blockIdx.x + (j / KB) * gridDim.x) * 128, jkb = j % KB;
                if (layout == 1)
                    prefetch_tile_l2(&tmA, 0, (blockIdx.x * tiles_per_cta * KB + j) * 128);
                else if (layout == 5 || layout == 7)
                    prefetch_tile_l2(&tmA, jkb * 128, jrow * 2);
                else if (layout == 6)
                    prefetch_tile_l2(&tmA, 0, (blockIdx.x * tiles_per_cta * KB + j) * 256);
                else
                    prefetch_tile_l2(&tmA, jkb * 128, jrow);
            }
            if (mode & 65536) {
                // bit 16: the producer polls the free barrier politely (a
                // 64 ns sleep between tests, bounded like mbar_wait)
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(b0 + 8 * (stages + s), ph ^ 1u)) {
                    if (*abort_flag || globaltimer() - t0 > 200000000ull) { ok = false; *abort_flag = 1; break; }
                    __nanosleep(64);
                }
                if (!ok) break;
            } else if (!mbar_wait(b0 + 8 * (stages + s), ph ^ 1u, 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; break; }
            mbar_arrive_expect_tx(b0 + 8 * s, box_tx + ((mode & 128) ? 1024u : 0u));
            if (blockIdx.x == 0 && i < 256) stamps[2 * i] = globaltimer();
            // bit 7: a second, 1 KB bulk copy per stage (a scale-atom pair) into the B area
            if (mode & 128)
                bulk_load(smem_u32(sm + stages * slot + 1024 * s), sf_src + ((size_t)blockIdx.x * total + i) * 1024,
                          1024, b0 + 8 * s);
            if (layout == 1)  // contiguous 8 KB tiles: 64-byte rows back to back
                tma_load_2d(smem_u32(sm + s * slot), &tmA, 0, (blockIdx.x * tiles_per_cta * KB + i) * 128, b0 + 8 * s);
            else if (layout == 3)  // 256-row fp4 box (two 128-row tiles per copy)
                tma_load_2d(smem_u32(sm + s * slot), &tmA, kb * 128, row, b0 + 8 * s);
            else if (layout == 5 || layout == 7)  // 256-row fp4 box, CTAs on disjoint 256-row tiles
                tma_load_2d(smem_u32(sm + s * slot), &tmA, kb * 128, row * 2, b0 + 8 * s);
            else if (layout == 6)  // contiguous 16 KB tiles: 256 rows of 64 bytes back to back
                tma_load_2d(smem_u32(sm + s * slot), &tmA, 0, (blockIdx.x * tiles_per_cta * KB + i) * 256, b0 + 8 * s);
            else
                tma_load_2d(smem_u32(sm + s * slot), &tmA, kb * 128, row, b0 + 8 * s);
        }
    } else if (warp == 2 && lane == 0 && (mode & 32768)) {
        // observer: the time each stage lands (it consumes nothing; on a
        // missed phase it stops observing)
        for (int i = 0; i < total && i < 256; ++i) {
            const int s = i % stages;
            const uint32_t ph = (uint32_t)((i / stages) & 1);
            if (!mbar_wait(b0 + 8 * s, ph, 5000000ull, abort_flag)) break;
            if (blockIdx.x == 0) stamps[768 + i] = globaltimer();
        }
    } else if (warp == 1 && lane == 0 && (mode & 262144)) {
        // bit 18: stages in groups of `pf` (1-4) -- wait for all of them,
        // then issue their MMAs (swapped operands, 4 per stage) and commits
        const int G = pf < 1 ? 1 : (pf > 4 ? 4 : pf);
        for (int i = 0; i < total && ok; i += G) {
            const int n = total - i < G ? total - i : G;
            for (int j = 0; j < n && ok; ++j) {
                const int s = (i + j) % stages;
                const uint32_t ph = (uint32_t)(((i + j) / stages) & 1);
                if (!mbar_wait(b0 + 8 * s, ph, 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; }
            }
            if (!ok) break;
            if (blockIdx.x == 0 && i < 256) stamps[2 * i + 1] = globaltimer();
            tc_fence_after();
            for (int j = 0; j < n; ++j) {
                const int s = (i + j) % stages;
                const uint32_t a = smem_u32(sm + s * slot), b = smem_u32(sm + stages * slot);
                for (int kk = 0; kk < 4; ++kk)
                    mma_mx(tmem, desc_sw128(b + 32 * kk), desc_sw128(a + 32 * kk),
                           idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk), tmem + 256, tmem + 260,
                           (kk > 0 || j > 0) ? 1u : 0u);
                mma_commit(b0 + 8 * (stages + s));
            }
        }
        if (ok) {
            mma_commit(b0 + 8 * (2 * stages + 1));
            if (!mbar_wait(b0 + 8 * (2 * stages + 1), 0, 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; }
        }
    } else if (warp == 1 && lane == 0) {
        for (int i = 0; i < total && ok; ++i) {
            const int s = i % stages;
            const uint32_t ph = (uint32_t)((i / stages) & 1);
            if (!mbar_wait(b0 + 8 * s, ph, 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; break; }
            if (blockIdx.x == 0 && i < 256) stamps[2 * i + 1] = globaltimer();
            if (mode & 16384) {
                // no MMAs: hold the slot for `pf` ns of wall time, then free it
                // (bit 17: free it first, then spin)
                if (mode & 131072) mbar_arrive(b0 + 8 * (stages + s));
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < (uint64_t)pf) {}
                if (blockIdx.x == 0 && i < 256) stamps[512 + i] = globaltimer();
                if (!(mode & 131072)) mbar_arrive(b0 + 8 * (stages + s));
                if (blockIdx.x == 0 && i < 256) stamps[1024 + i] = globaltimer();
                continue;
            }
            if (mode & 1) {
                // bit 2: no tcgen05 fence; bit 3: 16 MMAs per stage; bit 4: N = 128;
                // bit 5: unscaled kind::f8f6f4 instead of the block-scaled MMA;
                // bit 6: operands swapped (the weight tile as B, N = 256)
                // (mode bit 7, an extra 1 KB bulk copy per stage, is on the producer side)
                if (!(mode & 4)) tc_fence_after();
                const uint32_t a = smem_u32(sm + s * slot), b = smem_u32(sm + stages * slot);
                const uint32_t nn = (mode & 16) ? 128 : 32;
                const int reps = (mode & 8) ? 4 : 1;
                for (int rr = 0; rr < reps; ++rr)
                    for (int kk = 0; kk < 4; ++kk) {
                        if (mode & 64) {
                            // operands swapped: A = a fixed e4m3 tile (the token side), B = the
                            // streamed 256-row fp4 weight tile, N = 256: one MMA per K=32 step
                            // bit 8: the weight tile read through a no-swizzle
                            // descriptor (layout 7 writes it unswizzled; timing only)
                            // bit 11: the MMAs read a static 256-row tile instead of the
                            // landed stage (after the barrier and tail; timing only)
                            const uint32_t wt = (mode & 2048) ? smem_u32(sm + stages * slot + 16384 + 2048) : a;
                            const uint64_t bd = (mode & 256) ? smem_desc(wt + 32 * kk, 128, 1024, 0)
                                                             : desc_sw128(wt + 32 * kk);
                            // bit 9: the token operand one aliased 8-row group (no swizzle, stride 0)
                            const uint64_t ad = (mode & 512) ? smem_desc(b + 32 * kk, 16, 0, 0) : desc_sw128(b + 32 * kk);
                            // bit 10: the token operand in tensor memory (columns 384 + 8 kk)
                            if constexpr (kTA)
                                mma_mx_ta(tmem, tmem + 384 + 8 * kk, bd,
                                          idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk), tmem + 256, tmem + 260,
                                          (kk > 0 || rr > 0) ? 1u : 0u);
                            else
                            // bit 13: accumulate across stages (only the first MMA of the
                            // stream starts the accumulator), else each stage restarts it
                            mma_mx(tmem, ad, bd,
                                   idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk), tmem + 256, tmem + 260,
                                   (kk > 0 || rr > 0 || ((mode & 8192) && i > 0)) ? 1u : 0u);
                        } else if (mode & 32) {
                            const uint32_t id = (kFmtE2M1 << 7) | (kFmtE4M3 << 10) | ((nn >> 3) << 17) | (8u << 24) | (1u << 4);
                            asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                                         "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}"
                                         ::"r"(tmem), "l"(desc_sw128(a + 32 * kk)), "l"(desc_sw128(b + 32 * kk)), "r"(id),
                                           "r"((uint32_t)(kk > 0 || rr > 0)) : "memory");
                        } else {
                            mma_mx(tmem, desc_sw128(a + 32 * kk), desc_sw128(b + 32 * kk),
                                   idesc_mx(kFmtE2M1, kFmtE4M3, 128, nn, kk, kk), tmem + 128, tmem + 132,
                                   (kk > 0 || rr > 0) ? 1u : 0u);
                        }
                    }
                // stamps[512 + i]: the stage's MMAs and commit issued (CTA 0)
                if (blockIdx.x == 0 && i < 256) stamps[512 + i] = globaltimer();
                // bit 12 (with bit 11: the MMAs read no slot): free the slot
                // once its MMAs are issued, and commit to a barrier nobody waits on
                if (mode & 4096) {
                    mma_commit(b0 + 8 * (2 * stages));
                    mbar_arrive(b0 + 8 * (stages + s));
                } else {
                    mma_commit(b0 + 8 * (stages + s));
                }
            } else {
                mbar_arrive(b0 + 8 * (stages + s));
            }
        }
        // every MMA issued has completed before the tensor memory is freed
        if ((mode & 1) && ok) {
            mma_commit(b0 + 8 * (2 * stages + 1));
            if (!mbar_wait(b0 + 8 * (2 * stages + 1), 0, 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; }
        }
    }
    __syncthreads();
    if (*abort_flag) { spin_ns(200000); if (threadIdx.x == 0) atomicExch(ok_out, 0); }
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

// layout 0: fp4 [rows][4096] box 128x128 (rows 2 KB apart); 1: fp4 viewed as
// contiguous 64-byte rows (each box = 8 KB contiguous); 2: uint8 [rows][4096]
// box 128x128 (16 KB); 3: fp4 box 128 x 256 rows (16 KB of codes, 32 KB slot),
// neighbouring CTAs' boxes overlapping by 128 rows; 5: as 3 on disjoint
// 256-row tiles; 6: 256-row boxes over contiguous 16 KB tiles.
extern "C" int probe_stream(const uint8_t* a, long long rows, int grid, int tiles_per_cta, int stages, int mode,
                            int pf, unsigned long long* stamps, int* ok, float* ms, int layout) {
    CUtensorMap ta;
    int r;
    uint32_t tx = 8192, slot = 16384;
    if (layout == 1) r = make_map(&ta, a, 128, (uint64_t)rows * 32, 128, true);
    else if (layout == 2) { r = make_map(&ta, a, 4096, (uint64_t)rows / 2, 128, false); tx = 16384; }
    else if (layout == 3 || layout == 5) { r = make_map(&ta, a, 4096, (uint64_t)rows, 256, true); tx = 16384; slot = 32768; }
    else if (layout == 7) { r = make_map(&ta, a, 4096, (uint64_t)rows, 256, true, false); tx = 16384; slot = 32768; }
    else if (layout == 6) { r = make_map(&ta, a, 128, (uint64_t)rows * 32, 256, true); tx = 16384; slot = 32768; }
    else r = make_map(&ta, a, 4096, (uint64_t)rows, 128, true);
    if (r) return 1000 + r;
    const long long need = (long long)(grid * (tiles_per_cta - 1) + grid) * 128 + (layout == 3 ? 128 : 0);
    if (need > (layout == 2 ? rows / 2 : rows)) return 3;
    if (layout == 1 && (long long)grid * tiles_per_cta * 32 * 128 > rows * 32) return 4;
    if ((layout == 5 || layout == 7) && (long long)grid * tiles_per_cta * 256 > rows) return 4;
    if (layout == 6 && (long long)grid * tiles_per_cta * 32 * 256 > rows * 32) return 4;
    if (slot == 32768 && stages > 6) return 5;
    // tiles + B tile + barrier offset + barriers/slot + 1024 alignment slack
    const int smem = stages * (int)slot + 16384 + 1024 + 512 + 1024 + ((mode & 2048) ? 2048 + 32768 : 0);
    if (smem > 232448) return 8;
    if ((mode & 4096) && !(mode & 2048)) return 9;  // a slot freed early must not be read
    cudaFuncSetAttribute(k_stream<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_stream<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    // bit 7 reads 1 KB per stage from the start of the tensor (grid * tiles * 32 KB <= its size)
    if ((mode & 128) && (long long)grid * tiles_per_cta * 32 * 1024 > rows * 2048) return 6;
    if ((mode & 128) && stages * 1024 > 16384) return 7;
    if (mode & 1024)
        k_stream<true><<<grid, 96, smem>>>(ta, tiles_per_cta, 32, stages, mode, pf, stamps, ok, layout, tx, slot, a);
    else
        k_stream<false><<<grid, 96, smem>>>(ta, tiles_per_cta, 32, stages, mode, pf, stamps, ok, layout, tx, slot, a);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// The TMA weight stream (its consumer frees every stage at once) and an
// independent MMA loop on resident operands, side by side in one CTA per SM:
// does either engine slow the other when neither waits on the other's data?
// which: 1 the stream alone, 2 the MMAs alone, 3 both.  The stream moves
// 256-row fp4 boxes (16 KB of codes into 32 KB slots, 6 stages, CTAs on
// disjoint tiles); an MMA group is 4 block-scaled N = 256 MMAs (an aliased
// token A, a swizzled 256-row B) and a commit, two groups in flight.
// times[4 b ..]: stream start, stream end, MMA start, MMA end (ns).
__global__ void __launch_bounds__(96, 1)
k_stream_indep(const __grid_constant__ CUtensorMap tmA, int tiles_per_cta, int groups, int which,
               unsigned long long* times, int* ok_out) {
    constexpr int kStages = 6, kSlot = 32768, KB = 32;
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint8_t* bt = sm + kStages * kSlot;  // resident B (32 KB), then A (1 KB)
    uint8_t* at = bt + 32768;
    uint64_t* bars = reinterpret_cast<uint64_t*>(at + 1024);  // full[6], empty[6], mma[2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t b0 = smem_u32(bars), bm = b0 + 8 * 2 * kStages;
    for (int i = threadIdx.x; i < (32768 + 1024) / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(bt)[i] = 0x38383838u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2 * kStages + 2; ++s) mbar_init(b0 + 8 * s, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;
    const int total = tiles_per_cta * KB;
    unsigned long long* tm = times + 4 * (size_t)blockIdx.x;
    if (warp == 0 && lane == 0 && (which & 1)) {
        tm[0] = globaltimer();
        for (int i = 0; i < total && ok; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (uint32_t)((i / kStages) & 1);
            const int row = (blockIdx.x + (i / KB) * gridDim.x) * 128, kb = i % KB;
            if (!mbar_wait(b0 + 8 * (kStages + s), ph ^ 1u, 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; break; }
            mbar_arrive_expect_tx(b0 + 8 * s, 16384u);
            tma_load_2d(smem_u32(sm + s * kSlot), &tmA, kb * 128, row * 2, b0 + 8 * s);
        }
    } else if (warp == 1 && lane == 0 && (which & 1)) {
        for (int i = 0; i < total && ok; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (uint32_t)((i / kStages) & 1);
            if (!mbar_wait(b0 + 8 * s, ph, 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; break; }
            mbar_arrive(b0 + 8 * (kStages + s));
        }
        tm[1] = globaltimer();
    } else if (warp == 2 && lane == 0 && (which & 2)) {
        const uint32_t a = smem_u32(at), b = smem_u32(bt);
        tm[2] = globaltimer();
        for (int it = 0; it < groups && ok; ++it) {
            // (which bit 2: B is ring slot it % 6, whatever the stream is doing to it)
            const uint32_t bb = (which & 4) ? smem_u32(sm + (it % kStages) * kSlot) : b;
            // group it commits to barrier it % 2; before issuing it, wait for
            // group it - 2 (the previous commit to the same barrier)
            if (it >= 2 && !mbar_wait(bm + 8 * (it & 1), (uint32_t)(((it - 2) >> 1) & 1), 200000000ull, abort_flag)) {
                ok = false; *abort_flag = 1; break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_mx(tmem, smem_desc(a + 32 * kk, 16, 0, 0), desc_sw128(bb + 32 * kk),
                       idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk), tmem + 256, tmem + 260, (it | kk) ? 1u : 0u);
            mma_commit(bm + 8 * (it & 1));
        }
        for (int it = groups - 2 > 0 ? groups - 2 : 0; it < groups && ok; ++it)
            if (!mbar_wait(bm + 8 * (it & 1), (uint32_t)((it >> 1) & 1), 200000000ull, abort_flag)) { ok = false; *abort_flag = 1; }
        tm[3] = globaltimer();
    }
    __syncthreads();
    if (*abort_flag) { spin_ns(200000); if (threadIdx.x == 0) atomicExch(ok_out, 0); }
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

extern "C" int probe_stream_indep(const uint8_t* a, long long rows, int grid, int tiles_per_cta, int groups,
                                  int which, unsigned long long* times, int* ok, float* ms) {
    CUtensorMap ta;
    if (make_map(&ta, a, 4096, (uint64_t)rows, 256, true)) return 2;
    if ((long long)grid * tiles_per_cta * 256 > rows || groups < 2 || which < 1 || which > 7) return 3;
    const int smem = 6 * 32768 + 32768 + 1024 + 256 + 1024;
    cudaFuncSetAttribute(k_stream_indep, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    k_stream_indep<<<grid, 96, smem>>>(ta, tiles_per_cta, groups, which, times, ok);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// Cost of single-thread primitives in SM clock cycles (clock64), one CTA
// per SM: res[4 b + 0] a try_wait on a completed phase, [1] a test_wait on
// it, [2] a %globaltimer read, [3] an arrive on another barrier followed by
// a try_wait on the completed one.  park: where the rest of warp 0 is while
// lane 0 runs the loops -- 0 exited; 1 at the CTA barrier (with warp 1);
// 2 at a warp barrier; 3 running the same loops (converged warp); 4 at a
// warp shuffle.  Every lane of a warp meets the same barrier instruction
// (the CTA barrier is an aligned one).
__global__ void __launch_bounds__(64, 1) k_prim(int iters, int park, unsigned long long* res) {
    __shared__ __align__(8) uint64_t bars[2];
    const int lane = threadIdx.x & 31;
    const bool w0 = threadIdx.x < 32;
    if (park == 0 && (!w0 || lane != 0)) return;
    if ((park == 2 || park == 4) && !w0) return;
    const uint32_t b0 = smem_u32(&bars[0]), b1 = smem_u32(&bars[1]);
    if (w0 && lane == 0) {
        mbar_init(b0, 1);
        mbar_init(b1, (1 << 20) - 1);  // the largest count
        fence_mbar_init();
        mbar_arrive(b0);  // phase 0 of b0 completes
    }
    if (w0 && park != 0) __syncwarp();  // (park 0: lane 0 is alone in its warp)
    uint32_t acc = 0;
    unsigned long long g = 0;
    if (w0 && (lane == 0 || park == 3)) {
        unsigned long long* r = res + 4 * (size_t)blockIdx.x;
        long long t0 = clock64();
        for (int i = 0; i < iters; ++i) acc += mbar_try_wait(b0, 0) ? 1u : 0u;
        long long t1 = clock64();
        if (lane == 0) r[0] = (unsigned long long)(t1 - t0);
        t0 = clock64();
        for (int i = 0; i < iters; ++i) {
            uint32_t ok;
            asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                         "selp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(b0), "r"(0u) : "memory");
            acc += ok;
        }
        t1 = clock64();
        if (lane == 0) r[1] = (unsigned long long)(t1 - t0);
        t0 = clock64();
        for (int i = 0; i < iters; ++i) g += globaltimer();
        t1 = clock64();
        if (lane == 0) r[2] = (unsigned long long)(t1 - t0);
        t0 = clock64();
        for (int i = 0; i < iters; ++i) {  // b1 never completes (iters < its count)
            if (lane == 0) mbar_arrive(b1);
            acc += mbar_try_wait(b0, 0) ? 1u : 0u;
        }
        t1 = clock64();
        if (lane == 0) r[3] = (unsigned long long)(t1 - t0);
        if (acc == 0xFFFFFFFFu && g == 1) r[0] = 0;  // keep the loops
    }
    if (park == 4) acc = __shfl_sync(0xFFFFFFFFu, acc, 0);
    if (park == 2) __syncwarp();
    if (park == 1 || park == 3) __syncthreads();
    if (acc == 0xFFFFFFFEu) res[0] = 0;
}

extern "C" int probe_prim(int grid, int iters, int park, unsigned long long* res) {
    if (iters < 1 || iters >= (1 << 20) - 1) return 3;
    k_prim<<<grid, 64>>>(iters, park, res);
    return (int)cudaDeviceSynchronize();
}

// Plain HBM read stream: every thread sums 16-byte loads, grid-strided.
__global__ void k_read(const uint4* __restrict__ p, long long n, unsigned int* sink) {
    unsigned int acc = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const uint4 v = __ldcs(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x12345678u) atomicAdd(sink, 1u);
}

extern "C" int probe_read(const uint8_t* p, long long bytes, int grid, int block, unsigned int* sink, float* ms) {
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    k_read<<<grid, block>>>(reinterpret_cast<const uint4*>(p), bytes / 16, sink);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// Block-scaled MMA issue rate: one thread per CTA issues `iters` x 4 MMAs of
// M=128, N=n, K=32 (e2m1 or e4m3 A, e4m3 B) on shared-memory-resident tiles.
__global__ void __launch_bounds__(64, 1) k_mma_peak(int iters, int n, uint32_t a_fmt, int* ok_out) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 16384 + 32768);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x38383838u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) { mbar_init(smem_u32(bar), 1); *abort_flag = 0; fence_mbar_init(); }
    if (warp == 1) tmem_alloc(smem_u32(slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(sm), b = smem_u32(sm + 16384);
        for (int it = 0; it < iters; ++it)
            for (int kk = 0; kk < 4; ++kk)
                mma_mx(tmem, desc_sw128(a + 32 * kk), desc_sw128(b + 32 * kk),
                       idesc_mx(a_fmt, kFmtE4M3, 128, (uint32_t)n, kk, kk), tmem + 256, tmem + 260,
                       (it | kk) ? 1u : 0u);
        mma_commit(smem_u32(bar));
        if (!mbar_wait(smem_u32(bar), 0, 2000000000ull, abort_flag)) { atomicExch(ok_out, 0); spin_ns(200000); }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

extern "C" int probe_mma_peak(int grid, int iters, int n, uint32_t a_fmt, int* ok, float* ms) {
    const int smem = 16384 + 32768 + 1024 + 64;
    cudaFuncSetAttribute(k_mma_peak, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    k_mma_peak<<<grid, 64, smem>>>(iters, n, a_fmt, ok);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// Issue cost of the decode kernel's per-stage MMA group: per iteration `ncp`
// scale-factor copies (tcgen05.cp 32x128b.warpx4), four K=32 block-scaled
// MMAs on one or two accumulators (M = 128, N = n) and optionally one
// tcgen05.commit to an mbarrier nobody waits on.  Smem operands are fixed.
// mode: 0 as the grouped GEMMs issue them, 1 the same scale-factor ids for
// every kk, 2 the same operand addresses for every kk, 3 B read through the
// decode kernel's no-swizzle descriptor (16-byte K chunks 16 bytes apart),
// 4 the decode kernel's orientation (weights as the N = 256 B operand)
template <bool kTA>
__global__ void __launch_bounds__(64, 1) k_mma_mix(int iters, int n, int ncp, int commit, int acc2,
                                                  uint32_t a_fmt, int mode, int* ok_out) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    // A: 2 x 16 KB, B: 16 KB, SF atoms: 3 x 512 B, then barriers
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 49152 + 1536);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 49152 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x38383838u;
    for (int i = threadIdx.x; i < 1536 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm + 49152)[i] = 0x7F7F7F7Fu;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        mbar_init(smem_u32(bar + 1), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(sm), b = smem_u32(sm + 32768), sf = smem_u32(sm + 49152);
        for (int it = 0; it < iters; ++it) {
            if (mode >= 7) {
                // mode 7: the decode orientation with the weight tile (B) in
                // the no-swizzle K-major layout [K chunk][256 rows][16 B];
                // mode 8: A a real swizzled 128-row tile, B swizzled (the
                // grouped kernel's orientation); mode 9: as 8 with A in tensor
                // memory (columns 384 + 8 kk)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if constexpr (kTA) {
                        mma_mx_ta(tmem, tmem + 384 + 8 * kk, desc_sw128(a + 32 * kk),
                                  idesc_mx(kFmtE4M3, a_fmt, 128, 256, kk, kk), tmem + 256, tmem + 260,
                                  (it | kk) ? 1u : 0u);
                        continue;
                    }
                    const uint64_t ad = mode == 7 ? smem_desc(b + 32 * kk, 16, 0, 0) : desc_sw128(b + 32 * kk);
                    const uint64_t bd = mode == 7 ? smem_desc(a + 8192 * kk, 4096, 128, 0) : desc_sw128(a + 32 * kk);
                    mma_mx(tmem, ad, bd, idesc_mx(kFmtE4M3, a_fmt, 128, 256, kk, kk), tmem + 256, tmem + 260,
                           (it | kk) ? 1u : 0u);
                }
                if (commit) mma_commit(smem_u32(bar + 1));
                continue;
            }
            if (mode >= 5) {
                // the decode gate/up pattern: A's scales resident (column
                // 256), the weight tile's two scale atoms copied per stage
                // into stage-indexed columns; mode 5 copies them right before
                // the stage's MMAs, mode 6 one stage ahead (before the MMAs
                // of the previous stage)
                const uint32_t cur = tmem + 264 + 8 * (it & 1), nxt = tmem + 264 + 8 * ((it + 1) & 1);
                if (mode == 5 || it == 0) {
                    tmem_cp_32x128_x4(cur, desc_sf(sf));
                    tmem_cp_32x128_x4(cur + 4, desc_sf(sf + 512));
                }
                if (mode == 6 && it + 1 < iters) {
                    tmem_cp_32x128_x4(nxt, desc_sf(sf));
                    tmem_cp_32x128_x4(nxt + 4, desc_sf(sf + 512));
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_mx(tmem, smem_desc(b + 32 * kk, 16, 0, 0), desc_sw128(a + 32 * kk),
                           idesc_mx(kFmtE4M3, a_fmt, 128, 256, kk, kk), tmem + 256, cur, (it | kk) ? 1u : 0u);
                if (commit) mma_commit(smem_u32(bar + 1));
                continue;
            }
            for (int j = 0; j < ncp; ++j) tmem_cp_32x128_x4(tmem + 256 + 4 * j, desc_sf(sf + 512 * j));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t sid = mode == 1 ? 0u : (uint32_t)kk;
                const uint32_t ko = mode == 2 ? 0u : 32u * kk;
                const uint32_t id = idesc_mx(a_fmt, kFmtE4M3, 128, (uint32_t)n, sid, sid);
                // acc2 == 2: a separate accumulator per (row half, kk): eight
                // independent chains of N = 16 columns
                const uint32_t acc = (acc2 == 2) ? (it ? 1u : 0u) : ((it | kk) ? 1u : 0u);
                const uint32_t d0 = (acc2 == 2) ? tmem + 16 * kk : tmem;
                const uint32_t d1 = (acc2 == 2) ? tmem + 64 + 16 * kk : tmem + 128;
                if (mode == 4) {
                    // the decode kernel's orientation: A = one aliased token row
                    // (no swizzle, 8-row groups at stride 0), B = a 256-row
                    // weight tile, N = 256: one MMA per K=32 step
                    mma_mx(tmem, smem_desc(b + ko, 16, 0, 0), desc_sw128(a + ko),
                           idesc_mx(kFmtE4M3, a_fmt, 128, 256, kk, kk), tmem + 256, tmem + 260,
                           (it | kk) ? 1u : 0u);
                    continue;
                }
                const uint64_t bd = mode == 3 ? smem_desc(b + ko, 16, 128, 0) : desc_sw128(b + ko);
                mma_mx(d0, desc_sw128(a + ko), bd, id, tmem + 256, tmem + 264, acc);
                if (acc2) mma_mx(d1, desc_sw128(a + 16384 + ko), bd, id, tmem + 260, tmem + 264, acc);
            }
            if (commit) mma_commit(smem_u32(bar + 1));
        }
        mma_commit(smem_u32(bar));
        if (!mbar_wait(smem_u32(bar), 0, 2000000000ull, abort_flag)) { atomicExch(ok_out, 0); spin_ns(200000); }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

extern "C" int probe_mma_mix(int grid, int iters, int n, int ncp, int commit, int acc2, uint32_t a_fmt, int mode,
                             int* ok, float* ms) {
    if (n < 16 || n > (acc2 == 2 ? 16 : acc2 ? 128 : 256) || ncp < 0 || ncp > 3) return 3;
    const int smem = 49152 + 1536 + 1024 + 64;
    if (mode < 0 || mode > 9) return 3;
    cudaFuncSetAttribute(k_mma_mix<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_mma_mix<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    if (mode == 9)
        k_mma_mix<true><<<grid, 64, smem>>>(iters, n, ncp, commit, acc2, a_fmt, 8, ok);
    else
        k_mma_mix<false><<<grid, 64, smem>>>(iters, n, ncp, commit, acc2, a_fmt, mode, ok);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// The same stream with the fp4 tiles moved by 128 threads with 8-byte
// cp.async copies (no TMA) into the 16-byte-aligned unpacked layout (code
// group c of row r -> slot (c ^ (r % 8)) of the 128-byte row), completion
// tracked by cp.async.mbarrier.arrive.noinc on the stage's barrier.
__global__ void __launch_bounds__(160, 1)
k_stream_lsu(const uint8_t* __restrict__ w, int tiles_per_cta, int KB, int stages, unsigned long long* stamps,
             int* ok_out) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + stages * 16384);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * stages);
    const int warp = threadIdx.x >> 5;
    const uint32_t b0 = smem_u32(bars);
    if (threadIdx.x == 0) {
        for (int st = 0; st < stages; ++st) { mbar_init(b0 + 8 * st, 128); mbar_init(b0 + 8 * (stages + st), 1); }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int total = tiles_per_cta * KB;
    if (warp < 4) {
        const int t = threadIdx.x;
        for (int i = 0; i < total; ++i) {
            const int st = i % stages;
            const uint32_t ph = (uint32_t)((i / stages) & 1);
            const long long row0 = (long long)(blockIdx.x + (i / KB) * gridDim.x) * 128;
            const int kb = i % KB;
            if (!mbar_wait(b0 + 8 * (stages + st), ph ^ 1u, 200000000ull, abort_flag)) { *abort_flag = 1; break; }
            if (blockIdx.x == 0 && t == 0 && i < 256) stamps[2 * i] = globaltimer();
            const uint32_t dst0 = smem_u32(sm + st * 16384);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int idx = j * 128 + t, r = idx >> 3, c = idx & 7;
                const uint8_t* src = w + (row0 + r) * 2048 + kb * 64 + c * 8;
                const uint32_t dst = dst0 + r * 128 + ((c ^ (r & 7)) << 4);
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(b0 + 8 * st) : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (threadIdx.x == 128) {
        for (int i = 0; i < total; ++i) {
            const int st = i % stages;
            const uint32_t ph = (uint32_t)((i / stages) & 1);
            if (!mbar_wait(b0 + 8 * st, ph, 200000000ull, abort_flag)) { *abort_flag = 1; break; }
            if (blockIdx.x == 0 && i < 256) stamps[2 * i + 1] = globaltimer();
            mbar_arrive(b0 + 8 * (stages + st));
        }
    }
    __syncthreads();
    if (*abort_flag) { spin_ns(200000); if (threadIdx.x == 0) atomicExch(ok_out, 0); }
}

extern "C" int probe_stream_lsu(const uint8_t* a, long long rows, int grid, int tiles_per_cta, int stages,
                                unsigned long long* stamps, int* ok, float* ms) {
    if ((long long)(grid * (tiles_per_cta - 1) + grid) * 128 > rows) return 3;
    const int smem = stages * 16384 + 1024 + 16 * stages + 64;
    cudaFuncSetAttribute(k_stream_lsu, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    k_stream_lsu<<<grid, 160, smem>>>(a, tiles_per_cta, 32, stages, stamps, ok);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// Contention probe: warp 1 (lane 0) runs the decode kernel's MMA loop (four
// N = 256 block-scaled MMAs per iteration on resident operands) while warps
// 2-9 keep shared memory busy: load = 1 writes 16 bytes per thread per step
// into a 32 KB region (generic-proxy stores), load = 2 reads it, load = 0
// idles.  stamps[blockIdx.x] = the MMA loop's wall time (ns).
__global__ void __launch_bounds__(320, 1) k_contend(int iters, int load, unsigned long long* stamps, int* ok_out) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    // [0, 32K) weights (B), [32K, 48K) token tile (A), [48K, 49.5K) scale atoms,
    // [64K, 96K) the busy region, then barriers
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 98304);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 2);
    volatile int* stop = reinterpret_cast<volatile int*>(slot + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 2);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 98304 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x38383838u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        *stop = 0;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 32) {
        const uint32_t b = smem_u32(sm), a = smem_u32(sm + 32768), sf = smem_u32(sm + 49152);
        tmem_cp_32x128_x4(tmem + 256, desc_sf(sf));
        tmem_cp_32x128_x4(tmem + 260, desc_sf(sf + 512));
        tmem_cp_32x128_x4(tmem + 264, desc_sf(sf + 1024));
        const unsigned long long t0 = globaltimer();
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_mx(tmem, smem_desc(a + 32 * kk, 16, 0, 0), desc_sw128(b + 32 * kk),
                       idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk), tmem + 256, tmem + 260, (it | kk) ? 1u : 0u);
        }
        mma_commit(smem_u32(bar));
        const bool ok = mbar_wait(smem_u32(bar), 0, 2000000000ull, abort_flag);
        stamps[blockIdx.x] = globaltimer() - t0;
        if (!ok) atomicExch(ok_out, 0);
        *stop = 1;
    } else if (warp >= 2) {
        const int t = threadIdx.x - 64;
        uint4* busy = reinterpret_cast<uint4*>(sm + 65536);
        uint4 acc = make_uint4(0, 0, 0, 0);
        const unsigned long long t0 = globaltimer();
        for (int i = 0; !*stop && globaltimer() - t0 < 200000000ull; ++i) {
#pragma unroll 8
            for (int j = 0; j < 8; ++j) {
                const int idx = (t + 256 * ((i * 8 + j) & 7)) & 2047;  // 2048 x 16 B = 32 KB
                if (load == 1) {
                    busy[idx] = make_uint4(i, j, t, 0);
                } else if (load == 2) {
                    const uint4 v = busy[idx];
                    acc.x ^= v.x; acc.y += v.y;
                }
            }
        }
        if (acc.x == 0x12345678u) stamps[gridDim.x + blockIdx.x] = acc.y;  // keeps the reads
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

extern "C" int probe_contend(int grid, int iters, int load, unsigned long long* stamps, int* ok, float* ms) {
    const int smem = 98304 + 64 + 1024;
    cudaFuncSetAttribute(k_contend, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    k_contend<<<grid, 320, smem>>>(iters, load, stamps, ok);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

// Weight stream with the copies done by the load/store units instead of the
// TMA: warps 0-7 (one weight row per thread) load each 16 KB stage (256 rows
// x 64 bytes of packed fp4, plus the stage's 1 KB of scale atoms) into
// registers kLd stages ahead and store them into the 16-byte-slot, 128-byte-
// swizzled layout the MMA reads (8 data bytes per slot); warp 8 issues the
// decode kernel's MMAs (four N = 256 per stage, two scale copies) with
// mode & 1, else frees the stage at once.  Global layout: rows of 2048 bytes
// (K = 4096), CTA c streams rows [256 (c + G t), +256) x 32 K steps.
constexpr int kLd = 6;
__global__ void __launch_bounds__(320, 1)
k_stream_ldg(const __grid_constant__ CUtensorMap tmW, const uint8_t* __restrict__ w,
             const uint8_t* __restrict__ sf_src, int tiles_per_cta, int stages, int mode, int* ok_out) {
    // mode bit 1 (hybrid): odd stages are copied by the TMA (warp 9), even
    // stages by the load/store units; `stages` must then be even
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int slot = 32768 + 1024;  // padded weights + scale atoms
    uint8_t* tok = sm + stages * slot;  // 4 KB token area (A, aliased)
    uint64_t* bars = reinterpret_cast<uint64_t*>(tok + 4096);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * stages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t b0 = smem_u32(bars);
    for (int i = threadIdx.x; i < 4096 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(tok)[i] = 0x38383838u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(b0 + 8 * s, ((mode & 2) && (s & 1)) ? 1 : 256);
            mbar_init(b0 + 8 * (stages + s), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 9) tmem_alloc(smem_u32(tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int total = tiles_per_cta * 32;
    if (warp < 8) {
        // four lanes per row (16 bytes each, a row's 64 bytes contiguous):
        // thread p covers rows p / 4 + 64 j (j < 4), chunk c = p % 4
        const int p = threadIdx.x, c = p & 3, r0 = p >> 2;
        const int step = (mode & 2) ? 2 : 1;        // LSU stage j is global stage step * j
        const int n_lsu = (total + step - 1) / step;
        uint4 reg[kLd][4];
        uint4 sreg[kLd];
        auto load = [&](int i, int q) {
            const long long row0 = (long long)(blockIdx.x + (i / 32) * gridDim.x) * 256;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                reg[q][j] = __ldcs(reinterpret_cast<const uint4*>(w + (row0 + r0 + 64 * j) * 2048 + (i % 32) * 64) + c);
            if (p < 64) sreg[q] = __ldcs(reinterpret_cast<const uint4*>(sf_src + ((size_t)blockIdx.x * total + i) * 1024) + p);
        };
#pragma unroll
        for (int q = 0; q < kLd; ++q)
            if (q < n_lsu) load(step * q, q);
        bool run = true;
        for (int j0 = 0; j0 < n_lsu && run; j0 += kLd) {
#pragma unroll
            for (int q = 0; q < kLd; ++q) {  // compile-time register slot q
                const int j = j0 + q;
                if (j >= n_lsu) break;
                const int i = step * j;
                const int s = i % stages;
                const uint32_t ph = (uint32_t)((i / stages) & 1);
                if (!mbar_wait(b0 + 8 * (stages + s), ph ^ 1u, 200000000ull, abort_flag)) {
                    *abort_flag = 1;
                    run = false;
                    break;
                }
                uint8_t* st = sm + s * slot;
                // packed chunk c of row r holds 32 codes = element slots 2c, 2c + 1
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = r0 + 64 * j;
                    const uint32_t e0 = (2 * c) ^ (r & 7), e1 = (2 * c + 1) ^ (r & 7);
                    uint8_t* line = st + (r >> 3) * 1024 + (r & 7) * 128;
                    *reinterpret_cast<uint2*>(line + e0 * 16) = make_uint2(reg[q][j].x, reg[q][j].y);
                    *reinterpret_cast<uint2*>(line + e1 * 16) = make_uint2(reg[q][j].z, reg[q][j].w);
                }
                if (p < 64) reinterpret_cast<uint4*>(st + 32768)[p] = sreg[q];
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(b0 + 8 * s);
                if (j + kLd < n_lsu) load(step * (j + kLd), q);
            }
        }
    } else if (warp == 9 && lane == 0 && (mode & 2)) {
        // the TMA's share: the odd stages
        for (int i = 1; i < total; i += 2) {
            const int s = i % stages;
            const uint32_t ph = (uint32_t)((i / stages) & 1);
            if (!mbar_wait(b0 + 8 * (stages + s), ph ^ 1u, 200000000ull, abort_flag)) { *abort_flag = 1; break; }
            uint8_t* st = sm + s * slot;
            const uint32_t fb = b0 + 8 * s;
            mbar_arrive_expect_tx(fb, 16384u + 1024u);
            const int row = (blockIdx.x + (i / 32) * gridDim.x) * 256;
            tma_load_2d(smem_u32(st), &tmW, (i % 32) * 128, row, fb);
            bulk_load(smem_u32(st + 32768), sf_src + ((size_t)blockIdx.x * total + i) * 1024, 1024, fb);
        }
    } else if (warp == 8 && lane == 0) {
        const uint32_t a = smem_u32(tok);
        for (int i = 0; i < total; ++i) {
            const int s = i % stages;
            const uint32_t ph = (uint32_t)((i / stages) & 1);
            if (!mbar_wait(b0 + 8 * s, ph, 200000000ull, abort_flag)) { *abort_flag = 1; break; }
            if (mode & 1) {
                tc_fence_after();
                const uint32_t st = smem_u32(sm + s * slot);
                tmem_cp_32x128_x4(tmem + 260, desc_sf(st + 32768));
                tmem_cp_32x128_x4(tmem + 264, desc_sf(st + 32768 + 512));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_mx(tmem, smem_desc(a + 32 * kk, 16, 0, 0), desc_sw128(st + 32 * kk),
                           idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk), tmem + 256, tmem + 260, (i | kk) ? 1u : 0u);
                mma_commit(b0 + 8 * (stages + s));
            } else {
                mbar_arrive(b0 + 8 * (stages + s));
            }
        }
        if (mode & 1) {  // the last MMAs complete before the CTA frees its tensor memory
            const int s = (total - 1) % stages;
            mbar_wait(b0 + 8 * (stages + s), (uint32_t)(((total - 1) / stages) & 1), 200000000ull, abort_flag);
        }
    }
    __syncwarp();
    __syncthreads();
    if (*abort_flag) { spin_ns(200000); if (threadIdx.x == 0) atomicExch(ok_out, 0); }
    if (warp == 9) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

extern "C" int probe_stream_ldg(const uint8_t* w, long long bytes, const uint8_t* sf, long long sf_bytes, int grid,
                                int tiles_per_cta, int stages, int mode, int* ok, float* ms) {
    if ((long long)grid * tiles_per_cta * 256 * 2048 > bytes) return 3;
    if ((mode & 2) && (stages & 1)) return 8;
    CUtensorMap tw;
    if (int r = make_map(&tw, w, 4096, (uint64_t)(bytes / 2048), 256, true)) return 1000 + r;
    if ((long long)grid * tiles_per_cta * 32 * 1024 > sf_bytes) return 4;
    if (stages < 2 || stages > 6) return 5;
    const int smem = stages * (32768 + 1024) + 4096 + 16 * stages + 16 + 1024;
    cudaFuncSetAttribute(k_stream_ldg, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    k_stream_ldg<<<grid, 320, smem>>>(tw, w, sf, tiles_per_cta, stages, mode, ok);
    cudaEventRecord(e1);
    int rc = (int)cudaDeviceSynchronize();
    cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}
