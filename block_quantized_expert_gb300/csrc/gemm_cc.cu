// gemm_cc.cu -- grouped expert GEMMs on the CUDA cores (fp32 FMA over the
// exactly dequantised MXFP4 / NVFP4 / fp8 weights and MXFP8 activations).
//
// Weight kinds: 0 MXFP4 (e2m1, UE8M0 per 32), 1 fp8 e4m3 with 128x128 UE8M0
// tiles (the shared expert), 2 NVFP4-style (e2m1, e4m3 per 16, fp32 per
// matrix: CISM VALIDATION, "4-bit quantization scheme study", row "E2M1 +
// E4M3 b16"): a 32-block's two halves take their own scales and the matrix
// scale multiplies the finished dot product.
//
// Work item = (segment e, chunk of up to kChunk tokens of the segment,
// 32 output features).  The chunk's activation rows are dequantised once into
// shared memory; each warp streams one weight row at a time with 16-byte
// loads (lane l owns the 32-blocks l, l+32, ...), decodes it to fp32 in
// registers and reuses it for every token of the chunk; a warp-shuffle tree
// finishes each dot product.  Gate/up fuses SiLU(g)*u and the MXFP8
// requantisation of h (guide, section 4); down writes fp32 rows.
#include "common.cuh"
#include "layer.h"
#include "stage_event.h"

namespace moe {

struct CCArgs {
    int n_seg;
    const int32_t* counts;      // [n_seg]
    const int32_t* poff;        // [n_seg+1] padded row starts
    const int32_t* chunk_scan;  // [n_seg+1]
    const uint8_t *w1_q, *w1_s, *w2_q, *w2_s;
    const float *w1_g, *w2_g;   // kind 2: per-segment matrix scales [n_seg]
    const uint8_t* aq;          // activation codes [Rp][K]
    const uint8_t* as;          // activation scale atoms
    int K, N;                   // contraction length, output features
    uint8_t* hq;                // gate/up: [Rp][N] codes + atoms
    uint8_t* hs;
    float* y;                   // down: y[row][N]
    const int32_t* pos_row;     // down: padded position -> output row (null: identity)
};

constexpr int kCCThreads = 256;
constexpr int kCCWarps = kCCThreads / 32;

// 32 weights of block b of row `row` as fp32 (without the block scale).
template <int kWKind>
__device__ __forceinline__ void load_weight_block(const uint8_t* __restrict__ q, size_t row, int K,
                                                  int b, float* wv) {
    if (kWKind != 1) {  // MXFP4 / NVFP4: 16 bytes, even element in the low nibble
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(q + row * (size_t)(K / 2)) + b);
        const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int n = 0; n < 8; ++n) wv[8 * i + n] = e2m1_to_f32((wds[i] >> (4 * n)) & 15u);
    } else {            // fp8 e4m3: 32 bytes
        const uint4* p = reinterpret_cast<const uint4*>(q + row * (size_t)K + (size_t)b * 32);
        const uint4 r0 = __ldg(p), r1 = __ldg(p + 1);
        const uint32_t wds[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int n = 0; n < 4; ++n) wv[4 * i + n] = e4m3_to_f32((wds[i] >> (8 * n)) & 255u);
    }
}

// The block scale of 32-block b of row `row` (kind 2: of its first 16
// elements; weight_scale_hi: of its last 16).
template <int kWKind>
__device__ __forceinline__ float weight_scale(const uint8_t* __restrict__ s, size_t seg_row0,
                                              int row, int K, int b) {
    if (kWKind == 0) return ue8m0_to_f32(__ldg(s + (seg_row0 + row) * (size_t)(K / 32) + b));
    if (kWKind == 2) return e4m3_to_f32(__ldg(s + (seg_row0 + row) * (size_t)(K / 16) + 2 * b));
    return ue8m0_to_f32(__ldg(s + (size_t)(row / 128) * (K / 128) + b / 4));
}
__device__ __forceinline__ float weight_scale_hi(const uint8_t* __restrict__ s, size_t seg_row0, int row,
                                                 int K, int b) {
    return e4m3_to_f32(__ldg(s + (seg_row0 + row) * (size_t)(K / 16) + 2 * b + 1));
}

template <int kWKind, bool kGateUp>
__global__ void __launch_bounds__(kCCThreads) k_gemm_cc(CCArgs a) {
    extern __shared__ float smem[];
    pdl_launch_dependents();
    pdl_wait();
    float* xf = smem;                          // [kChunk][K]
    float* hb = smem + kChunk * a.K;           // [kChunk][32]
    __shared__ float lut8[256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int c = threadIdx.x; c < 256; c += kCCThreads) lut8[c] = e4m3_to_f32(c);

    const int total = __ldg(a.chunk_scan + a.n_seg) * (a.N / 32);
    const int KB = a.K / 32;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const int chunk = item / (a.N / 32), fb = item % (a.N / 32);
        int lo = 0, hi = a.n_seg;  // segment e with chunk_scan[e] <= chunk < chunk_scan[e+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(a.chunk_scan + mid) <= chunk) lo = mid; else hi = mid;
        }
        const int e = lo;
        const int n0 = (chunk - __ldg(a.chunk_scan + e)) * kChunk;
        const int nt = min(kChunk, __ldg(a.counts + e) - n0);
        const int p0 = __ldg(a.poff + e) + n0;

        __syncthreads();  // previous item done with xf / hb
        for (int i = threadIdx.x; i < nt * a.K; i += kCCThreads) {
            const int n = i / a.K, h = i % a.K;
            const float sc = ue8m0_to_f32(a.as[sf_atom_offset(p0 + n, h / 32, a.K)]);
            xf[n * a.K + h] = lut8[a.aq[(size_t)(p0 + n) * a.K + h]] * sc;
        }
        __syncthreads();

        const size_t seg_row0 = (kWKind != 1) ? (size_t)e * a.N : 0;
        for (int jj = warp; jj < 32; jj += kCCWarps) {
            const int j = fb * 32 + jj;
            float acc1[kChunk], acc2[kChunk];
#pragma unroll
            for (int n = 0; n < kChunk; ++n) { acc1[n] = 0.f; acc2[n] = 0.f; }
            // gate/up codes are interleaved per 128 features (gate block, then up
            // block); down codes are row-major per segment
            const size_t prow = kGateUp ? (size_t)((kWKind != 1 ? e : 0) * (a.N / 128) + j / 128) * 256 + (j % 128)
                                        : seg_row0 + j;
            for (int b = lane; b < KB; b += 32) {
                float w1[32];
                load_weight_block<kWKind>(a.w1_q, prow, a.K, b, w1);
                const float s1 = weight_scale<kWKind>(a.w1_s, seg_row0, j, a.K, b);
                const float s1h = kWKind == 2 ? weight_scale_hi(a.w1_s, seg_row0, j, a.K, b) : s1;
                float w2[32];
                float s2 = 0.f, s2h = 0.f;
                if (kGateUp) {
                    load_weight_block<kWKind>(a.w2_q, prow + 128, a.K, b, w2);
                    s2 = weight_scale<kWKind>(a.w2_s, seg_row0, j, a.K, b);
                    s2h = kWKind == 2 ? weight_scale_hi(a.w2_s, seg_row0, j, a.K, b) : s2;
                }
#pragma unroll
                for (int n = 0; n < kChunk; ++n) {
                    if (n < nt) {
                        const float4* xv = reinterpret_cast<const float4*>(xf + n * a.K + b * 32);
                        // the two 16-element halves (one scale each for kind 2)
                        float p1[2] = {0.f, 0.f}, p2[2] = {0.f, 0.f};
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 x4 = xv[i];
                            float& q1 = p1[i >> 2];
                            q1 = fmaf(w1[4 * i], x4.x, q1); q1 = fmaf(w1[4 * i + 1], x4.y, q1);
                            q1 = fmaf(w1[4 * i + 2], x4.z, q1); q1 = fmaf(w1[4 * i + 3], x4.w, q1);
                            if (kGateUp) {
                                float& q2 = p2[i >> 2];
                                q2 = fmaf(w2[4 * i], x4.x, q2); q2 = fmaf(w2[4 * i + 1], x4.y, q2);
                                q2 = fmaf(w2[4 * i + 2], x4.z, q2); q2 = fmaf(w2[4 * i + 3], x4.w, q2);
                            }
                        }
                        if (kWKind == 2) {
                            acc1[n] = fmaf(p1[1], s1h, fmaf(p1[0], s1, acc1[n]));
                            if (kGateUp) acc2[n] = fmaf(p2[1], s2h, fmaf(p2[0], s2, acc2[n]));
                        } else {
                            acc1[n] = fmaf(p1[0] + p1[1], s1, acc1[n]);
                            if (kGateUp) acc2[n] = fmaf(p2[0] + p2[1], s2, acc2[n]);
                        }
                    }
                }
            }
            // kind 2: the matrix scales multiply the finished dot products
            const float g1 = kWKind == 2 ? __ldg(a.w1_g + e) : 1.f;
            const float g2 = (kWKind == 2 && kGateUp) ? __ldg(a.w2_g + e) : 1.f;
#pragma unroll
            for (int n = 0; n < kChunk; ++n) {
                const float g = warp_sum(acc1[n]) * g1;
                if (kGateUp) {
                    const float u = warp_sum(acc2[n]) * g2;
                    if (lane == 0 && n < nt) hb[n * 32 + jj] = silu_mul(g, u);
                } else {
                    if (lane == 0 && n < nt) hb[n * 32 + jj] = g;
                }
            }
        }
        __syncthreads();

        if (warp < nt) {  // one warp per token of the chunk
            const int n = warp, p = p0 + n;
            const float v = hb[n * 32 + lane];
            if (kGateUp) {
                const float amax = warp_max(fabsf(v));
                const int ex = mxfp8_exponent(amax);
                const uint32_t code = f32x2_to_e4m3x2(scale_pow2(v, ex), 0.f) & 0xFFu;
                a.hq[(size_t)p * a.N + fb * 32 + lane] = (uint8_t)code;
                if (lane == 0) a.hs[sf_atom_offset(p, fb, a.N)] = (uint8_t)(ex + 127);
            } else {
                const int row = a.pos_row ? __ldg(a.pos_row + p) : p;
                if (row >= 0) a.y[(size_t)row * a.N + fb * 32 + lane] = v;
            }
        }
    }
}

cudaError_t cc_init() {
    const int smem = (int)(sizeof(float) * kChunk * (8192 + 32));  // K <= 8192: 131.6 KB
    cudaError_t e = cudaFuncSetAttribute(k_gemm_cc<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_cc<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_cc<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_cc<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_cc<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_cc<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return e;  // the dynamic smem request already selects the largest carveout
}

template <int kWKind, bool kGateUp>
static cudaError_t cc_launch(moe_layer* L, const CCArgs& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * (size_t)kChunk * (a.K + 32);
    const int grid = L->num_sms * 2;
    L->launches += 1;
    return launch_pdl(k_gemm_cc<kWKind, kGateUp>, dim3(grid), dim3(kCCThreads), smem, s, a);
}

cudaError_t launch_gemm_cc(moe_layer* L, int T, cudaStream_t s, cudaEvent_t mid) {
    (void)T;
    const moe_config& c = L->cfg;
    CCArgs a{};
    // routed experts: gate/up over H, then down over I
    a.n_seg = c.n_experts;
    a.counts = L->counts;
    a.poff = L->poff;
    a.chunk_scan = L->chunk_scan;
    a.w1_q = L->gu_q; a.w1_s = L->gate_s; a.w2_q = L->gu_q; a.w2_s = L->up_s;
    a.w1_g = L->gate_g; a.w2_g = L->up_g;
    a.aq = L->xq; a.as = L->xs;
    a.K = c.hidden; a.N = c.inter;
    a.hq = L->hq; a.hs = L->hs;
    const bool nv = c.weight_format == MOE_WEIGHTS_NVFP4;
    cudaError_t err = nv ? cc_launch<2, true>(L, a, s) : cc_launch<0, true>(L, a, s);
    if (err == cudaSuccess && mid) err = record_stage(mid, s);
    if (err != cudaSuccess) return err;
    CCArgs d = a;
    d.w1_q = L->down_q; d.w1_s = L->down_s; d.w2_q = nullptr; d.w2_s = nullptr;
    d.w1_g = L->down_g; d.w2_g = nullptr;
    d.aq = L->hq; d.as = L->hs;
    d.K = c.inter; d.N = c.hidden;
    d.y = L->y; d.pos_row = L->pos_row;
    err = nv ? cc_launch<2, false>(L, d, s) : cc_launch<0, false>(L, d, s);
    if (err != cudaSuccess || !c.has_shared) return err;
    // shared expert: one segment of all T tokens in token order
    CCArgs sg{};
    sg.n_seg = 1;
    sg.counts = L->sh_desc; sg.poff = L->sh_desc + 1; sg.chunk_scan = L->sh_desc + 5;
    sg.w1_q = L->sh_gu_q; sg.w1_s = L->sh_gate_s; sg.w2_q = L->sh_gu_q; sg.w2_s = L->sh_up_s;
    sg.aq = L->xq_tok; sg.as = L->xs_tok;
    sg.K = c.hidden; sg.N = c.inter;
    sg.hq = L->hq_sh; sg.hs = L->hs_sh;
    err = cc_launch<1, true>(L, sg, s);
    if (err != cudaSuccess) return err;
    CCArgs sd = sg;
    sd.w1_q = L->sh_down_q; sd.w1_s = L->sh_down_s; sd.w2_q = nullptr; sd.w2_s = nullptr;
    sd.aq = L->hq_sh; sd.as = L->hs_sh;
    sd.K = c.inter; sd.N = c.hidden;
    sd.y = L->y_sh; sd.pos_row = nullptr;
    return cc_launch<1, false>(L, sd, s);
}

}  // namespace moe
