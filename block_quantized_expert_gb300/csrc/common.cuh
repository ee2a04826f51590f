// common.cuh -- device helpers shared by the libmoe kernels: number formats,
// the block-scale layout of activations, warp reductions and error flags.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp8.h>
#include <cstdint>

#include "../../include/moe.h"

namespace moe {

// Sticky device error flags (bit set in layer->d_err).
enum : uint32_t { ERR_BAD_ID = 1u, ERR_TIMEOUT = 2u };

constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 1024;
constexpr int kRowTile = 128;   // permuted segments start at multiples of this

// ---------------------------------------------------------------- formats --
// e2m1 value of a 4-bit code: 1 sign, 2 exponent (bias 1), 1 mantissa bit.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
    uint32_t mag = c & 7u;
    uint32_t bits = (mag < 2u) ? (mag ? 0x3F000000u : 0u)                    // 0, 0.5
                               : (((mag >> 1) + 126u) << 23) | ((mag & 1u) << 22);
    return __uint_as_float(bits | ((c & 8u) << 28));
}

// e4m3 (fn) value of a byte: bias 7, subnormals m * 2^-9, S.1111.111 = NaN.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    uint32_t e = (c >> 3) & 15u, m = c & 7u;
    float mag;
    if (e == 15u && m == 7u) mag = __uint_as_float(0x7FC00000u);
    else if (e == 0u) mag = (float)m * 0.001953125f;                          // 2^-9
    else mag = __uint_as_float(((e + 120u) << 23) | (m << 20));             // 2^(e-7)(1+m/8)
    return (c & 0x80u) ? -mag : mag;
}

// UE8M0 byte -> 2^(c-127) (c = 0 gives the fp32 subnormal 2^-127).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t c) {
    return c ? __uint_as_float(c << 23) : __uint_as_float(0x00400000u);
}

// MXFP8 scale exponent of a 32-block from its amax (exact, from the fp32
// exponent field): floor(log2 amax) - 8 clamped to [-127, 127]; amax = 0 or
// an fp32 subnormal amax (floor(log2) <= -127) gives -127.
__device__ __forceinline__ int mxfp8_exponent(float amax) {
    int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
    int ex = ef - 127 - 8;
    return (ef == 0 || ex < -127) ? -127 : ex;   // ef <= 254 keeps ex <= 119
}

// v * 2^-ex for the exponents mxfp8_exponent returns (-127 <= ex <= 119):
// 2^-ex is a normal fp32 built from its exponent field, so the product is
// one IEEE multiplication (rounded once, as a scaling by a power of two is).
__device__ __forceinline__ float scale_pow2(float v, int ex) {
    return v * __uint_as_float((uint32_t)(127 - ex) << 23);
}

// Two fp32 -> two e4m3 bytes (round to nearest even, saturate to +-448),
// first value in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// ------------------------------------------------- activation scale layout --
// Block scales of activations (rows x K, one byte per 32-block) are stored in
// 512-byte atoms, one per (128-row tile, 128-column tile): inside an atom the
// byte of (row r, block kk) is at (r % 32) * 16 + (r / 32) * 4 + kk, the
// order the tcgen05 block-scaled MMA wants after a 32x128b.warpx4 copy.
__device__ __host__ __forceinline__ size_t sf_atom_offset(int row, int kb, int K) {
    int rt = row >> 7, r = row & 127;
    return ((size_t)rt * (size_t)(K >> 7) + (size_t)(kb >> 2)) * 512u +
           (size_t)((r & 31) * 16 + (r >> 5) * 4 + (kb & 3));
}

// ------------------------------------------------------------------ warps --
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ void raise_flag(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Programmatic dependent launch: allow the next kernel of the stream to be
// scheduled now (its prologue overlaps this kernel), and wait until the
// previous kernel has completed and its writes are visible.  Every kernel
// waits before its first global access, so stream order is kept.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ unsigned long long tc_globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t) :: "memory");  // not moved across barriers
    return t;
}

}  // namespace moe
