/*
 * moe_peaks.h -- C ABI of libmoe_peaks: the measured denominators of the
 * layer's rooflines.  Not part of the layer: the bench and the peak tool
 * call it to put each kernel's achieved rate beside what this GPU does.
 *
 * The routed-expert layer's decode and pp512 kernels are weight-read streams
 * bound by HBM ("DeepSeek-V4-Flash 284B - Deep-Dive Mathematical & Kernel
 * Guide", section 2A: decode time is the MUL_MAT_ID weight reads); the 8192-
 * token prefill is bound by the block-scaled tensor cores, and the CUDA-core
 * decode kernel's arithmetic runs barely above the HBM rate.  Each entry point
 * runs on the current CUDA device, synchronises the device, and returns a
 * cudaError_t code (0 = success).  No allocation is made; the caller owns
 * every pointer.
 */
#ifndef MOE_PEAKS_H
#define MOE_PEAKS_H

#ifdef __cplusplus
extern "C" {
#endif

/* Read `bytes` (>= 16, a multiple of 16) of device memory at p (16-byte
 * aligned) once, with `grid` blocks of 512 threads issuing 16-byte loads.
 * sink: one device uint32 the kernel may increment (keeps the loads live).
 * *ms (host): the kernel's duration from CUDA events.  Invalid arguments
 * return cudaErrorInvalidValue before any launch. */
int peak_read_stream(const void* p, long long bytes, int grid, unsigned int* sink, float* ms);

/* `grid` CTAs (use one per SM) each issue iters x 4 block-scaled MMAs
 * (tcgen05.mma kind::mxf8f6f4, scale_vec::1X, M 128, N 256, K 32, e4m3 A x
 * e2m1 B: 2*128*256*32 flops each) on operands resident in shared memory.
 * ok: one device int32 the caller sets to 1; a CTA whose bounded final wait
 * (2 s) gave up writes 0.  *ms (host): the kernel's duration. */
int peak_mma_mx(int grid, int iters, int* ok, float* ms);

/* The arithmetic of the CUDA-core decode kernel without its memory traffic:
 * `grid` CTAs of 16 warps each run `iters` iterations in which every warp
 * takes four 32-blocks of e2m1 codes from shared memory (one per lane, 4 x
 * 1024 elements a warp), converts the code pairs to f16 (cvt.rn.f16x2.e2m1x2)
 * and multiplies them by f16 operands with fp32 accumulation
 * (fma.rn.f32.f16).  seed: 1024 device uint32 (codes and operands);
 * out: grid x 512 device floats (keeps the sums live); cyc: grid device
 * int64, each CTA's loop in SM clock cycles, so that elements per clock per
 * SM = iters x 16 x 4 x 1024 / cyc.  *ms (host): the kernel's duration. */
int peak_dot_e2m1(int grid, int iters, const unsigned int* seed, float* out, long long* cyc, float* ms);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PEAKS_H */
