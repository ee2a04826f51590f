// decode_gemv.cu -- the whole layer for one token (T = 1) as a split-K GEMV on
// the CUDA cores: the fp4 weights stream into shared memory by bulk copies,
// the e2m1 codes are decoded by the hardware converter, their products with
// the MXFP8 token are summed in fp32 and reduced across the warp by shuffles.
// One cooperative kernel, one CTA per SM: routing, quantisation, gate/up,
// SwiGLU + MXFP8 requantisation of h, down and the fixed-order combine.
//
// Why the CUDA cores.  With one token the tensor-core MMA does 1/128 useful
// work, and the tcgen05 kernel's stream of weight copies and MMAs runs at
// ~0.5 us per 16 KB stage per SM.  The e2m1 -> f16x2 converter and the mixed
// f16 x f16 + f32 FMA (half rate) do ~59 elements per clock per SM (the
// peak_dot_e2m1 measurement), about 1.4 times what HBM delivers per SM, so a
// lean stage loop keeps up with the copies.
//
// Arithmetic of one 32-block (the block-scaled dot product of the method):
// the e2m1 weight values and the e4m3 values of the token (or of h) are
// exact in f16, so each product is exact in fp32; the block's 32 products are
// summed in fp32 (four partial sums of 8), the sum is multiplied by the two
// UE8M0 block scales (powers of two), and the blocks' values of a row are
// summed across the lanes of the warp.  NVFP4-style weights: each 16-element
// half's sum is multiplied by its own e4m3 scale, and the matrix scales
// multiply the finished dot products.
//
// Work split (the same in every CTA, from the kept count m and the grid G):
//  * gate/up: the m * I / 32 "h blocks" (32 consecutive features of one
//    expert: 32 gate rows + the 32 matching up rows, K = H) go to the CTAs
//    round-robin, block b to CTA b mod G.  A CTA owns whole blocks, so it
//    forms h = SiLU(g) * u and its MXFP8 requantisation (32 features share
//    a scale) itself.
//  * down: each CTA owns a contiguous range of d output rows (a multiple of
//    4) for every kept expert, so out[o] = sum over experts (ascending) of
//    w_s * y_s[o] is formed in the CTA that computed the y_s[o]: no combine
//    pass, no atomics.  The ranges are sized so that every CTA streams about
//    the same bytes (gate/up blocks + down rows).
//  * a CTA streams its work as stages of 32 KB of codes (+ their rows' scale
//    bytes): RG = 65536 / H rows of a block's gate or up half, or RD = 65536 /
//    I down rows, the CTA's (expert, row) pairs in order -- a stage may span
//    experts, in runs of 4 rows.  A producer warp bulk-copies them into a
//    ring of kStages buffers; 16 compute warps each take 4 consecutive rows
//    of one K segment (4 x 512 bytes: one 32-block per lane), whose operand
//    (the token, or h) they hold in registers as f16.  The down weights do
//    not depend on h: the producer streams on while h is exchanged, and
//    starts before the routing weights are known when the kept count does
//    not depend on them.
//  * h exchange: a publisher warp (which first computes the routing
//    weights) publishes each of the CTA's h blocks once the compute warps'
//    partial sums of it are in, as 6 64-bit words tagged with the launch's
//    epoch (a reader that sees the tag sees the payload: one L2 round trip,
//    no flags); two gatherer warps poll the kept experts' words, two experts
//    a pass, and copy them into shared memory for the compute warps.
// Cross-CTA hand-offs carry the launch's epoch: CTA c counts its own
// launches in a word of its own (read at the start, advanced at the exit;
// every CTA of a grid runs once per launch, so all hold the same count), so
// nothing is ever reset, no CTA contends for a counter, and graph replays
// get fresh epochs.
#include <cuda_fp8.h>

#include <cstdint>
#include <new>

#include "common.cuh"
#include "layer.h"
#include "route.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace gemv {

using tc::bulk_load;
using tc::globaltimer;
using tc::mbar_arrive;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::smem_u32;

constexpr int kComputeWarps = 16;
constexpr int kProducer = kComputeWarps;      // warp index: bulk copies into the ring (lane 0)
constexpr int kService = kComputeWarps + 1;   // warp index: routing weights, publishing the CTA's h blocks
constexpr int kGather = kComputeWarps + 2;    // warp indices kGather, kGather + 1: gathering the kept experts' h
constexpr int kThreads = 32 * (kComputeWarps + 4);
constexpr int kSeg = 1024;                    // K elements of one warp step (32 lanes x one 32-block)
constexpr int kRun = 4;                       // consecutive rows of a compute warp in a stage
constexpr int kStageCodes = 512 * kRun * kComputeWarps;  // bytes of codes per stage (32 KB)
// the rows' scale bytes of a stage: one per 32-block (MXFP4: UE8M0), two
// (NVFP4: an e4m3 scale per 16 elements)
__host__ __device__ constexpr int stage_scales(bool nv) { return kStageCodes / (nv ? 8 : 16); }
__host__ __device__ constexpr int stage_bytes(bool nv) { return kStageCodes + stage_scales(nv); }
constexpr int kStages = 5;
constexpr int kMaxK = kMaxTopK;
constexpr int kMaxPos = kMaxK + 1;            // kept positions: the routed experts, then the shared expert
constexpr int kRunS = 2;                      // rows of a compute warp in a stage of fp8 (shared-expert) rows
constexpr int kMaxI = 4096;                   // (the h words of every position are resident in shared memory)
// A published h block (32 features): 6 64-bit words, word w holding e4m3 codes
// 6w .. 6w + 5 in bytes 0 .. 5 (the last word: codes 30, 31 and the block's
// scale byte in byte 2) and the low 8 bits of the launch's epoch in byte 7
// (a single-copy atomic store: a reader that sees the tag sees the payload).
// Every launch writes every block of its k (+ 1 with the shared expert)
// positions -- published, or (positions after the m kept ones and the shared
// one) overwritten with a payload no reader uses -- so a word older than the
// launch carries the previous launch's tag, never this one's.
constexpr int kHWords = 6;
constexpr int kGatherWords = 12;             // words a gather lane has in flight

struct Args {
    const float* logits;  // [E]
    const uint16_t* x;    // [H] bf16 (device, or mapped host memory when x_stage is set)
    int E, k, H, I;
    float w_scale;
    RoutePrune prune;
    int32_t* ids_out;  // [k]
    float* w_out;      // [k]
    float* out;        // [H]
    const uint8_t* gu_q;    // [E][I/128][gate 128 rows, up 128 rows][H/2]
    const uint8_t* gate_s;  // [E][I][H/32] (NVFP4: [E][I][H/16] e4m3)
    const uint8_t* up_s;    // [E][I][H/32] (NVFP4: [E][I][H/16] e4m3)
    const uint8_t* down_q;  // [E][H][I/2]
    const uint8_t* down_s;  // [E][H][I/32] (NVFP4: [E][H][I/16] e4m3)
    const float *gate_g, *up_g, *down_g;  // NVFP4: the per-expert matrix scales [E]
    // the shared expert (sh set): e4m3 codes, gate/up interleaved per 128
    // features [I/128][256][H], down [H][I]; UE8M0 scales per 128 x 128 tile
    int sh;
    const uint8_t *sh_gu_q, *sh_gate_s, *sh_up_s, *sh_down_q, *sh_down_s;
    unsigned long long* hw;  // [kMaxPos][I/32][kHWords]: h by kept position, epoch-tagged words
    uint32_t* launches;     // [G]: launches CTA c has completed (its epoch - 1)
    uint16_t* x_stage;      // CTA 0's device copy of a host x, or null
    uint32_t* x_flag;       // x_stage written (the launch's epoch)
    uint32_t* err;
    uint64_t wait_ns;       // wall-time limit of every wait
    int stall_h;            // test hook: the h waits expect a value no CTA writes
    int nbmax, dmax;        // the largest h-block count and down range of a CTA (smem sizing)
    int RG, RD, spb;        // rows per gate/up and per down stage, stages per h block
    int RGs, RDs, spbs;     // the same for the shared expert's fp8 rows
    const int32_t* rows;    // [k][G + 1]: CTA c's down rows [rows[c], rows[c + 1]) for m = 1 .. k kept
    unsigned long long* trace;  // diagnostics (see stamp / trace_event), or null
};

// ------------------------------------------------------------- work split --
// Output rows [cut[x], cut[x + 1]) of CTA x (x = 0 .. G - 1), so that the
// CTAs' stream bytes are about equal.  The h blocks -- m * I / 32 routed ones,
// then I / 32 of the shared expert -- go to CTA b mod G; a CTA's capacity for
// down rows is max(0, W / G - its gate/up bytes) (W = all bytes), the H rows
// are cut in proportion to the capacities (prefix sums, so the ranges tile
// [0, H) in CTA order), and every cut is rounded to a multiple of 4 rows (H is
// one).  Host only: the kernel reads the table.
inline void split_rows(int G, int m, int H, int I, bool nv, bool sh, int* cut) {
    const long long sb = nv ? 16 : 32;  // elements per weight scale byte
    const long long FB = I / 32, NBr = (long long)m * FB, NB = NBr + (sh ? FB : 0);
    const long long Wr = 64LL * (H / 2 + H / sb), Ws = 64LL * H;  // a routed / the shared expert's h block
    const long long Wdn = (long long)m * (I / 2 + I / sb) + (sh ? I : 0);  // one output row of every expert
    const long long Wg = (NBr * Wr + (NB - NBr) * Ws + (long long)H * Wdn) / G;
    auto cap = [&](long long x) {
        const long long nr = x < NBr ? (NBr - 1 - x) / G + 1 : 0, nt = x < NB ? (NB - 1 - x) / G + 1 : 0;
        const long long gu = nr * Wr + (nt - nr) * Ws;
        return Wg > gu ? Wg - gu : 0;
    };
    long long total = 0;
    for (long long x = 0; x < G; ++x) total += cap(x);
    long long pre = 0;
    for (long long x = 0; x < G; ++x) {
        const long long r = total <= 0 ? x * H / G : H * pre / total;
        cut[x] = (int)((r + 2) / 4 * 4);
        if (cut[x] > H) cut[x] = H;
        pre += cap(x);
    }
    cut[G] = H;
}

// Shared-memory layout (bytes), the same on the host and the device.
struct Layout {
    int ring, route, lg, bars, pgu, pdn, hraw, shs, total;
    __host__ __device__ Layout(int H, int I, int nbmax, int dmax, bool nv, bool sh) {
        const int NQ = H / kSeg, NQd = I / kSeg;
        ring = 0;                                     // [kStages][stage_bytes(nv)]
        route = ring + kStages * stage_bytes(nv);     // sel, w_t, seg_e, seg_w, prod_e [8] each; words [16]
        lg = route + 256;                             // the logits [E <= 1024], candidates [256] x 2
        const int np = sh ? kMaxPos : kMaxK;          // positions with h: the kept experts (+ the shared one)
        bars = lg + 4096 + 2048;  // full [kStages], empty [kStages], blk [nbmax], h_ready [kMaxPos]
        pgu = bars + ((8 * (2 * kStages + nbmax + kMaxPos) + 15) / 16) * 16;  // [nbmax][NQ][64] f32
        pdn = pgu + nbmax * NQ * 64 * 4;              // [np][NQd][dmax] f32
        hraw = pdn + ((np * NQd * dmax * 4 + 15) / 16) * 16;  // [np][I/32][kHWords] h words as published
        shs = hraw + np * (I / 32) * kHWords * 8;     // the shared expert's tile scales: gate, up, down
        total = shs + (sh ? ((3 * (I / 128) * (H / 128) + 15) / 16) * 16 : 0);
    }
};
// words of the route area
enum { W_M = 0, W_EPOCH = 1, W_ABORT = 2 };

// ------------------------------------------------------------- arithmetic --
// One 32-bit word of e2m1 codes (elements 8i .. 8i + 7 of a block, the even
// element in the low nibble) -> four f16x2, element 2j in the low half of o[j].
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n.reg .b8 b0, b1, b2, b3;\nmov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\ncvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\ncvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}
// Two e4m3 bytes (the first in the low byte) -> f16x2 (the first in the low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
// acc + lo(a) lo(b) + hi(a) hi(b): f16 operands, each product exact in fp32,
// fp32 sums (low half first).
__device__ __forceinline__ float dot2_f16_f32(uint32_t a, uint32_t b, float acc) {
    asm("{\n.reg .b16 al, ah, bl, bh;\nmov.b32 {al, ah}, %1;\nmov.b32 {bl, bh}, %2;\n"
        "fma.rn.f32.f16 %0, al, bl, %0;\nfma.rn.f32.f16 %0, ah, bh, %0;\n}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}
// The block's dot product: 16 bytes of e2m1 codes against op (f16x2 of the
// block's 32 operand values, elements 2j, 2j + 1 in op[j]); four partial
// sums over the block's four 8-element quarters, returned as the two
// 16-element halves' sums (q0 + q1, q2 + q3).
__device__ __forceinline__ float2 block_dot_halves(const uint4& w, const uint32_t (&op)[16]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h[4];
        e2m1x8_to_f16x2(ws[i], h);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i] = dot2_f16_f32(h[j], op[4 * i + j], acc[i]);
    }
    return make_float2(acc[0] + acc[1], acc[2] + acc[3]);
}
// The block's dot product for e4m3 weight codes (the shared expert): 32
// bytes (two 16-byte loads) against op, four partial sums of 8.
__device__ __forceinline__ float block_dot_fp8(const uint4& w0, const uint4& w1, const uint32_t (&op)[16]) {
    const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        acc[i >> 1] = dot2_f16_f32(e4m3x2_to_f16x2(ws[i]), op[2 * i], acc[i >> 1]);
        acc[i >> 1] = dot2_f16_f32(e4m3x2_to_f16x2(ws[i] >> 16), op[2 * i + 1], acc[i >> 1]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}
// The operand of a down run: a lane's published h block (6 tagged words): its
// codes as f16 pairs, its scale from the last word.
__device__ __forceinline__ void load_h(const unsigned long long* hp, uint32_t (&op)[16], float& opsf) {
#pragma unroll
    for (int w = 0; w < 5; ++w) {
        const unsigned long long hv = hp[w];
        op[3 * w] = e4m3x2_to_f16x2((uint32_t)hv);
        op[3 * w + 1] = e4m3x2_to_f16x2((uint32_t)(hv >> 16));
        op[3 * w + 2] = e4m3x2_to_f16x2((uint32_t)(hv >> 32));
    }
    const unsigned long long h5 = hp[5];
    op[15] = e4m3x2_to_f16x2((uint32_t)h5);
    opsf = ue8m0_to_f32((uint32_t)(h5 >> 16) & 0xFFu);
}
// Two e4m3 scale bytes (the first in the low byte) -> fp32.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    return make_float2(__half2float(__half(__half_raw{h.x})), __half2float(__half(__half_raw{h.y})));
}
// A row's 32-block value times its weight scale(s): MXFP4 (one UE8M0 byte in
// sv) (lo + hi) * 2^s; NVFP4 (two e4m3 bytes) lo * s0 + hi * s1.
template <bool kNv>
__device__ __forceinline__ float scaled_block(const uint4& w, const uint32_t (&op)[16], uint32_t sv) {
    const float2 d = block_dot_halves(w, op);
    if (kNv) {
        const float2 sc = e4m3x2_to_f32x2(sv);
        return fmaf(d.y, sc.y, d.x * sc.x);
    }
    return (d.x + d.y) * ue8m0_to_f32(sv);
}
// One lane's 32-block of the token (16 words of bf16 pairs) -> MXFP8 (the
// block's scale 2^ex from its amax, e4m3 codes rounded to nearest even) ->
// the codes' values as f16x2 in op, the scale as fp32 in sf.
__device__ __forceinline__ void quantize_token(const uint32_t (&xw)[16], uint32_t (&op)[16], float& sf) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(xw[i] << 16)), fabsf(__uint_as_float(xw[i] & 0xFFFF0000u))));
    const int ex = mxfp8_exponent(amax);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t two = f32x2_to_e4m3x2(scale_pow2(__uint_as_float(xw[i] << 16), ex),
                                             scale_pow2(__uint_as_float(xw[i] & 0xFFFF0000u), ex));
        op[i] = e4m3x2_to_f16x2(two);
    }
    sf = ue8m0_to_f32((uint32_t)(ex + 127));
}
// Four per-lane values summed over the warp: afterwards lane l holds the
// total of value 2 * ((l >> 4) & 1) + ((l >> 3) & 1) (lanes 0, 8, 16, 24:
// values 0, 1, 2, 3).
__device__ __forceinline__ float warp_sum4(float v0, float v1, float v2, float v3, int lane) {
    const bool b4 = lane & 16, b3 = lane & 8;
    const float a = (b4 ? v2 : v0) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? v0 : v2, 16);
    const float b = (b4 ? v3 : v1) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? v1 : v3, 16);
    float r = (b3 ? b : a) + __shfl_xor_sync(0xFFFFFFFFu, b3 ? a : b, 8);
#pragma unroll
    for (int o = 4; o; o >>= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
    return r;
}

// ------------------------------------------------------------------ sync --
// Publish / await an epoch flag (release / acquire at gpu scope).
__device__ __forceinline__ void flag_set(uint32_t* f, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t flag_get(const uint32_t* f) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
__device__ __forceinline__ void st_tagged(unsigned long long* p, unsigned long long payload, uint32_t epoch) {
    const unsigned long long v = ((unsigned long long)(epoch & 0xFFu) << 56) | payload;
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ bool flag_wait(const uint32_t* f, uint32_t v, volatile int* abort, uint64_t limit_ns) {
    if (flag_get(f) == v) return true;
    const uint64_t t0 = globaltimer();
    while (flag_get(f) != v) {
        if (globaltimer() - t0 > limit_ns || *abort) return false;
        __nanosleep(64);
    }
    return true;
}

// Diagnostics (a.trace set): per CTA c, trace[8 c + slot] = wall-clock ns of
// slot 0 entry, 2 publisher done, 3 first kept expert's h gathered, 4 first
// copy issued, 5 final barrier; and for CTAs 0, 1, 80 and G - 1 (t = 0 .. 3)
// an event record at trace[8 G + 256 t + i]: i = 128 + stage (copy issued),
// 192 + j (h block j's partials in), 200 + j (published), 208 + s (kept
// expert s gathered).
__device__ __forceinline__ void stamp(const Args& a, int slot) {
    if (a.trace) a.trace[(size_t)blockIdx.x * 8 + slot] = globaltimer();
}
__device__ __forceinline__ void trace_event(const Args& a, int i) {
    const int c = blockIdx.x, G = gridDim.x;
    const int t = c == 0 ? 0 : c == 1 ? 1 : c == 80 ? 2 : c == G - 1 ? 3 : -1;
    if (a.trace && t >= 0 && i < 256) a.trace[(size_t)G * 8 + 256 * t + i] = globaltimer();
}
// --------------------------------------------------------------- stages --
// The CTA's stages, in stream order: for each of its nb h blocks (j), the
// block's gate rows then its up rows, RG rows a stage; then the CTA's down
// rows of every kept expert, as the flat list u = s * d + o (s ascending, o
// the row in [r0, r0 + d)), RD rows a stage.
struct Plan {
    int c, G, FB, H, I, m, nb, nbr, r0, d;
    int RG, RD, spb, RGs, RDs, spbs;  // rows per gate/up and per down stage, stages per h block (routed, shared)
    int ngur, ngu, ndr, n;            // stages: routed gate/up, all gate/up, + routed down, all
};
template <bool kSh>
__device__ __forceinline__ void make_plan(Plan& p, const Args& a, int c, int G, int m, const int32_t* cuts) {
    p.c = c;
    p.G = G;
    p.FB = a.I / 32;
    p.H = a.H;
    p.I = a.I;
    p.m = m;
    const int NBr = m * p.FB, NB = NBr + (kSh ? p.FB : 0);
    p.nbr = c < NBr ? (NBr - c + G - 1) / G : 0;  // this CTA's h blocks: c, c + G, .. (routed first)
    p.nb = c < NB ? (NB - c + G - 1) / G : 0;
    p.r0 = cuts[2 * (m - 1)];
    p.d = cuts[2 * (m - 1) + 1] - p.r0;
    p.RG = a.RG;
    p.RD = a.RD;
    p.spb = a.spb;
    p.RGs = a.RGs;
    p.RDs = a.RDs;
    p.spbs = a.spbs;
    p.ngur = p.nbr * p.spb;
    p.ngu = p.ngur + (p.nb - p.nbr) * p.spbs;
    p.ndr = p.ngu + (m * p.d + p.RD - 1) / p.RD;
    p.n = p.ndr + (kSh ? (p.d + p.RDs - 1) / p.RDs : 0);
}
// (producer) The copies of stage i into the ring buffer at dst, completing on
// the barrier fb: one contiguous run of codes and one of scale bytes per
// expert the stage's rows belong to.
template <bool kNv, bool kSh>
__device__ __forceinline__ void issue_stage(const Args& a, const Plan& p, const int* seg_e, int i, uint8_t* dst,
                                            uint32_t fb) {
    constexpr int SB = kNv ? 16 : 32;  // elements per scale byte
    if (kSh && i >= p.ngur && i < p.ngu) {
        // a shared-expert gate/up stage: RGs fp8 rows of block j (scales: in shared memory)
        const int i2 = i - p.ngur, j2 = i2 / p.spbs, row0 = (i2 - j2 * p.spbs) * p.RGs;
        const int fb32 = p.c + (p.nbr + j2) * p.G - p.m * p.FB;
        const int f = 32 * fb32 + (row0 & 31), up = row0 >> 5;
        const size_t grow = (size_t)(f >> 7) * 256 + up * 128 + (f & 127);
        const uint32_t cb = (uint32_t)(p.RGs * p.H);
        mbar_arrive_expect_tx(fb, cb);
        bulk_load(smem_u32(dst), a.sh_gu_q + grow * p.H, cb, fb);
    } else if (kSh && i >= p.ndr) {
        // a shared-expert down stage: up to RDs fp8 rows of the CTA's range
        const int u0 = (i - p.ndr) * p.RDs, u1 = min(u0 + p.RDs, p.d);
        const uint32_t cb = (uint32_t)((u1 - u0) * p.I);
        mbar_arrive_expect_tx(fb, cb);
        bulk_load(smem_u32(dst), a.sh_down_q + (size_t)(p.r0 + u0) * p.I, cb, fb);
    } else if (i < p.ngur) {
        const int j = i / p.spb, row0 = (i - j * p.spb) * p.RG;
        const int b = p.c + j * p.G, s = b / p.FB, fb32 = b - s * p.FB;
        const int e = seg_e[s], f = 32 * fb32 + (row0 & 31), up = row0 >> 5;
        const size_t grow = ((size_t)e * (p.I / 128) + (f >> 7)) * 256 + up * 128 + (f & 127);
        const uint32_t cb = (uint32_t)(p.RG * (p.H / 2)), sb = (uint32_t)(p.RG * (p.H / SB));
        mbar_arrive_expect_tx(fb, cb + sb);
        bulk_load(smem_u32(dst), a.gu_q + grow * (p.H / 2), cb, fb);
        bulk_load(smem_u32(dst + kStageCodes), (up ? a.up_s : a.gate_s) + ((size_t)e * p.I + f) * (p.H / SB), sb, fb);
    } else {
        const int u0 = (i - p.ngu) * p.RD, u1 = min(u0 + p.RD, p.m * p.d);  // (routed down)
        mbar_arrive_expect_tx(fb, (uint32_t)(u1 - u0) * (uint32_t)(p.I / 2 + p.I / SB));
        for (int u = u0; u < u1;) {
            const int s = u / p.d, o = u - s * p.d, n = min(u1 - u, p.d - o);
            const size_t drow = (size_t)seg_e[s] * p.H + p.r0 + o;
            bulk_load(smem_u32(dst + (u - u0) * (p.I / 2)), a.down_q + drow * (p.I / 2), (uint32_t)(n * (p.I / 2)), fb);
            bulk_load(smem_u32(dst + kStageCodes + (u - u0) * (p.I / SB)), a.down_s + drow * (p.I / SB),
                      (uint32_t)(n * (p.I / SB)), fb);
            u += n;
        }
    }
}

// One warp publishes a finished h block of this CTA (block j of the CTA,
// global block b of kept expert s): g and u summed over the K segments in
// order, h = SiLU(g) * u, MXFP8 over the 32 features (lane f: feature
// 32 fb + f), then the block's tagged words: lane 4w stores codes 4w .. 4w + 3
// (the first in the low byte), lane 0 the scale byte.
template <bool kNv>
__device__ void publish_block(const Args& a, const float* pgu, const int* seg_e, int m, int j, int b, int FB,
                              int NQ, uint32_t epoch, int lane) {
    const int s = b / FB, fb = b - s * FB;
    float g = 0.f, u = 0.f;
    for (int q = 0; q < NQ; ++q) {
        g += pgu[(j * NQ + q) * 64 + lane];
        u += pgu[(j * NQ + q) * 64 + 32 + lane];
    }
    if (kNv && b < m * FB) {  // (routed) the matrix scales multiply the finished dot products
        g *= __ldg(a.gate_g + seg_e[s]);
        u *= __ldg(a.up_g + seg_e[s]);
    }
    const float h = silu_mul(g, u);
    const int ex = mxfp8_exponent(warp_max(fabsf(h)));
    const uint32_t code = f32x2_to_e4m3x2(scale_pow2(h, ex), 0.f) & 0xFFu;
    // lane 6w collects codes 6w .. 6w + 5 (lane 30: codes 30, 31 and the scale)
    unsigned long long word = code;
#pragma unroll
    for (int i = 1; i < 6; ++i) {
        const unsigned long long ci = __shfl_down_sync(0xFFFFFFFFu, code, i);
        if (lane + i < 32) word |= ci << (8 * i);
    }
    if (lane == 30) word |= (unsigned long long)(ex + 127) << 16;
    unsigned long long* dst = a.hw + ((size_t)s * FB + fb) * kHWords;
    if (lane % 6 == 0 && lane <= 30) st_tagged(dst + lane / 6, word, epoch);
}

// 20 warps: 16 compute warps, the producer, the publisher and two gatherers
// (at most 96 registers a thread: 5 warps on one SM quarter).
template <bool kNv, bool kSh>
__global__ void __launch_bounds__(kThreads, 1) k_decode_gemv(const __grid_constant__ Args a) {
    constexpr int kStageBytes = stage_bytes(kNv), kSB = kNv ? 16 : 32;  // (kSB: elements per scale byte)
    extern __shared__ __align__(128) uint8_t smem[];
    const Layout Lo(a.H, a.I, a.nbmax, a.dmax, kNv, kSh);
    int* sel = reinterpret_cast<int*>(smem + Lo.route);  // [8] the router's selection, in router order
    float* w_t = reinterpret_cast<float*>(sel + 8);
    int* seg_e = reinterpret_cast<int*>(w_t + 8);         // [8] the kept experts, ascending
    float* seg_w = reinterpret_cast<float*>(seg_e + 8);   // [8] their weights
    int* prod_e = reinterpret_cast<int*>(seg_w + 8);      // [8] the producer's copy of seg_e
    volatile int* words = reinterpret_cast<volatile int*>(prod_e + 8);
    volatile int* abort_flag = words + W_ABORT;
    int32_t* cuts = reinterpret_cast<int32_t*>(prod_e + 8) + 4;  // [8][2] (after the words)
    float* lg = reinterpret_cast<float*>(smem + Lo.lg);
    const uint32_t full0 = smem_u32(smem + Lo.bars), empty0 = full0 + 8u * kStages;
    const uint32_t blk0 = empty0 + 8u * kStages, hrdy0 = blk0 + 8u * a.nbmax;
    float* pgu = reinterpret_cast<float*>(smem + Lo.pgu);
    float* pdn = reinterpret_cast<float*>(smem + Lo.pdn);
    unsigned long long* hraw = reinterpret_cast<unsigned long long*>(smem + Lo.hraw);
    uint8_t* shs = smem + Lo.shs;  // the shared expert's tile scales: gate, up [I/128][H/128], down [H/128][I/128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int NQ = a.H / kSeg, NQd = a.I / kSeg, FB = a.I / 32;
    const int qx = warp % NQ, qh = warp % NQd;  // (compute warps) K segments of the token and of h

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(full0 + 8u * st, 1);
            mbar_init(empty0 + 8u * st, kComputeWarps);
        }
        for (int j = 0; j < a.nbmax; ++j) mbar_init(blk0 + 8u * j, kComputeWarps);
        for (int s = 0; s < kMaxPos; ++s) mbar_init(hrdy0 + 8u * s, 64);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (threadIdx.x < 8) sel[threadIdx.x] = -1;
    pdl_launch_dependents();
    pdl_wait();
    stamp(a, 0);
    if (kSh) {  // the shared expert's tile scales (3 x (I/128)(H/128) bytes), in place before the routing barrier
        const int nt = (a.I / 128) * (a.H / 128);
        for (int i = threadIdx.x; i < 3 * nt; i += kThreads)
            shs[i] = i < nt ? __ldg(a.sh_gate_s + i) : i < 2 * nt ? __ldg(a.sh_up_s + i - nt) : __ldg(a.sh_down_s + i - 2 * nt);
    }
    // (producer lanes j < k) CTA c's down-row cuts for j + 1 kept experts,
    // in flight during the routing
    if (warp == kProducer && lane < a.k) {
        cuts[2 * lane] = __ldg(a.rows + (size_t)lane * (G + 1) + c);
        cuts[2 * lane + 1] = __ldg(a.rows + (size_t)lane * (G + 1) + c + 1);
    }
    uint32_t n_launch = 0;
    if (threadIdx.x == 32) n_launch = *reinterpret_cast<volatile uint32_t*>(a.launches + c);
    // ---- routing, first round: warp w ranks the 32 logits of chunk w (and
    // w + 19, ..) among themselves and keeps its local top k as candidates
    // -- every global top-k logit is one (larger logit first, equal logits to
    // the lower index, NaN never selected: the selection of route_token)
    int* ci = reinterpret_cast<int*>(lg + 1024);  // [<= 256] candidate experts (-1: none)
    float* cv = lg + 1024 + 256;                   // [<= 256] their logits (NaN: none)
    const int nchunk = (a.E + 31) / 32, nc = nchunk * a.k;  // nc <= 32 * 8
    for (int chk = warp; chk < nchunk; chk += kThreads / 32) {
        const int e = chk * 32 + lane;
        const float v = e < a.E ? __ldg(a.logits + e) : __int_as_float(0x7FC00000);
        if (e < a.E) lg[e] = v;
        int r = 0;
#pragma unroll
        for (int l2 = 0; l2 < 32; ++l2) {
            const float u = __shfl_sync(0xFFFFFFFFu, v, l2);
            r += (u > v || (u == v && l2 < lane)) ? 1 : 0;
        }
        if (lane < a.k) {
            ci[chk * a.k + lane] = -1;
            cv[chk * a.k + lane] = __int_as_float(0x7FC00000);
        }
        __syncwarp();
        if (v == v && r < a.k) {
            ci[chk * a.k + r] = e;
            cv[chk * a.k + r] = v;
        }
    }
    // (padding) the candidate slots up to a multiple of 4 are empty
    if (threadIdx.x < (-nc & 3)) {
        ci[nc + threadIdx.x] = -1;
        cv[nc + threadIdx.x] = __int_as_float(0x7FC00000);
    }
    // (compute warps) the token's segment qx, one 32-block per lane, from a
    // device x: loaded now, quantised once the copies are issued (a host x is
    // staged by CTA 0 after the routing)
    uint32_t op[16];
    float opsf = 0.f;
    uint32_t xw[16];
    if (warp < kComputeWarps && !a.x_stage) {
        const uint4* xp = reinterpret_cast<const uint4*>(a.x + qx * kSeg + 32 * lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = __ldg(xp + i);
            xw[4 * i] = v.x;
            xw[4 * i + 1] = v.y;
            xw[4 * i + 2] = v.z;
            xw[4 * i + 3] = v.w;
        }
    }
    __syncthreads();
    // second round: thread t ranks candidate t among all candidates (four at
    // a time; empty slots hold NaN: never counted)
    for (int t = threadIdx.x; t < nc; t += kThreads) {
        const int e = ci[t];
        if (e < 0) continue;
        const float v = cv[t];
        int r = 0;
#pragma unroll 4
        for (int t2 = 0; t2 < nc; t2 += 4) {
            const float4 u = *reinterpret_cast<const float4*>(cv + t2);
            const int4 ie = *reinterpret_cast<const int4*>(ci + t2);
            r += (int)(u.x > v) | ((int)(u.x == v) & (int)(ie.x < e));
            r += (int)(u.y > v) | ((int)(u.y == v) & (int)(ie.y < e));
            r += (int)(u.z > v) | ((int)(u.z == v) & (int)(ie.z < e));
            r += (int)(u.w > v) | ((int)(u.w == v) & (int)(ie.w < e));
        }
        if (r < a.k) sel[r] = e;
    }
    if (threadIdx.x == 32) words[W_EPOCH] = (int)(n_launch + 1u);
    __syncthreads();
    const uint32_t epoch = (uint32_t)words[W_EPOCH];

    if (warp == kProducer) {
        // ------------------------------------------------------ producer
        // Without pruning the kept experts are the router's k (every
        // selection valid), known now: the first ring's worth of copies (free
        // slots: no wait; lane i issues stage i) starts before the routing
        // weights; the rest after the barrier that publishes them.
        const bool early = !prunes(a.prune, a.k);
        int m = 0, i0 = 0;
        Plan p;
        if (early) {
            const int e = lane < a.k ? sel[lane] : 0;
            m = __all_sync(0xFFFFFFFFu, e >= 0) ? a.k : 0;
            int pos = 0;
            for (int j = 0; j < m; ++j) pos += (__shfl_sync(0xFFFFFFFFu, e, j) < e) ? 1 : 0;
            if (lane < m) prod_e[pos] = e;
            __syncwarp();
            if (m > 0) {
                make_plan<kSh>(p, a, c, G, m, cuts);
                i0 = min(p.n, kStages);
                if (lane < i0) {
                    issue_stage<kNv, kSh>(a, p, prod_e, lane, smem + Lo.ring + lane * kStageBytes, full0 + 8u * lane);
                    trace_event(a, 128 + lane);
                }
                if (lane == 0) stamp(a, 4);
            }
        }
        __syncthreads();  // (the routing weights)
        if (!early) {
            m = words[W_M];
            if (lane < m) prod_e[lane] = seg_e[lane];
            __syncwarp();
            if (m > 0) make_plan<kSh>(p, a, c, G, m, cuts);
        }
        if (m > 0 && lane == 0) {
            int slot = i0 % kStages;
            uint32_t par = (uint32_t)(((i0 / kStages) & 1) ^ 1);
            for (int i = i0; i < p.n; ++i) {
                if (!mbar_wait(empty0 + 8u * slot, par, a.wait_ns, abort_flag) || *abort_flag) {
                    *abort_flag = 1;
                    raise_flag(a.err, ERR_TIMEOUT);
                    break;
                }
                if (i == 0) stamp(a, 4);
                issue_stage<kNv, kSh>(a, p, prod_e, i, smem + Lo.ring + slot * kStageBytes, full0 + 8u * slot);
                trace_event(a, 128 + i);
                if (++slot == kStages) {
                    slot = 0;
                    par ^= 1u;
                }
            }
        }
        __syncwarp();
    } else {
        if (warp < kComputeWarps && !a.x_stage) quantize_token(xw, op, opsf);
        if (warp == kService) {
            // the routing weights (the arithmetic of route_token: w_j =
            // w_scale * s_j / (s_0 + .. + s_{k-1}), s = sqrt(softplus(logit)),
            // then the tail pruning) and the kept experts in ascending order
            const int k = a.k;
            int e = lane < k ? sel[lane] : 0;
            const bool ok = __all_sync(0xFFFFFFFFu, e >= 0);
            float sv = 0.f;
            if (lane < k && ok) sv = sqrt_softplus(lg[e]);
            float sum = 0.f;
            for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xFFFFFFFFu, sv, j));
            float wj = (lane < k && ok) ? route_weight(a.w_scale, sv, sum) : 0.0f;
            const int m = !ok ? 0 : (prunes(a.prune, k) ? prune_tail(wj, k, a.prune, lane) : k);
            int pos = 0;
            for (int j = 0; j < m; ++j) pos += (__shfl_sync(0xFFFFFFFFu, e, j) < e) ? 1 : 0;
            if (lane < m) {
                seg_e[pos] = e;
                seg_w[pos] = wj;
            }
            if (c == 0 && lane < k) {
                a.ids_out[lane] = lane < m ? e : -1;  // (pruned slots: -1, weight 0)
                a.w_out[lane] = wj;
            }
            if (c == 0 && lane == 0 && !ok) raise_flag(a.err, ERR_BAD_ID);
            if (lane == 0) words[W_M] = m;
        } else if (warp < kComputeWarps && a.x_stage) {
            // a host x: through CTA 0's device copy
            constexpr int kCT = 32 * kComputeWarps;
            if (c == 0) {
                for (int i = threadIdx.x; i < a.H / 8; i += kCT)
                    reinterpret_cast<uint4*>(a.x_stage)[i] = reinterpret_cast<const uint4*>(a.x)[i];
                asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory");
                if (threadIdx.x == 0) flag_set(a.x_flag, epoch);
            } else {
                if (threadIdx.x == 0 && !flag_wait(a.x_flag, epoch, abort_flag, a.wait_ns)) {
                    *abort_flag = 1;
                    raise_flag(a.err, ERR_TIMEOUT);
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory");
            }
            const uint4* xp = reinterpret_cast<const uint4*>(a.x_stage + qx * kSeg + 32 * lane);
            uint32_t xw[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = __ldcg(xp + i);
                xw[4 * i] = v.x;
                xw[4 * i + 1] = v.y;
                xw[4 * i + 2] = v.z;
                xw[4 * i + 3] = v.w;
            }
            quantize_token(xw, op, opsf);
        }
        __syncthreads();  // (the routing weights)
    }
    const int m = words[W_M];
    const int mp = m > 0 ? m + (kSh ? 1 : 0) : 0;  // positions with h this launch: the kept experts, then the shared one
    if (warp == kService) {
        // blocks of the positions mp .. k + sh - 1 (round-robin like the
        // published ones): their words get this launch's tag, so that no word
        // is ever more than one launch old
        const unsigned long long inval = 0;
        for (int b = mp * FB + ((c - mp * FB) % G + G) % G; b < (a.k + (kSh ? 1 : 0)) * FB; b += G)
            if (lane < kHWords) st_tagged(a.hw + (size_t)b * kHWords + lane, inval, epoch);
    }
    if (m == 0) {
        // no valid routing (ERR_BAD_ID is raised): the output is zero
        for (int i = c * kThreads + threadIdx.x; i < a.H; i += G * kThreads) a.out[i] = 0.f;
        __syncthreads();
        if (threadIdx.x == 0) a.launches[c] = epoch;
        return;
    }
    Plan p;
    make_plan<kSh>(p, a, c, G, m, cuts);

    if (warp == kService) {
        // ------------------------------------------------------ publisher
        // the CTA's h blocks, each once every compute warp has stored its
        // partials of it
        bool ok = true;
        for (int j = 0; j < p.nb && ok; ++j) {
            if (!mbar_wait(blk0 + 8u * j, 0, a.wait_ns, abort_flag)) {
                ok = false;
                break;
            }
            if (lane == 0) trace_event(a, 192 + j);
            publish_block<kNv>(a, pgu, seg_e, m, j, c + j * G, FB, NQ, epoch, lane);
            if (lane == 0) trace_event(a, 200 + j);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            raise_flag(a.err, ERR_TIMEOUT);
        }
        if (lane == 0) stamp(a, 2);
    } else if (warp == kGather || warp == kGather + 1) {
        // ------------------------------------------------------ gatherers
        // the kept experts' h, P experts a pass: the pass's words (positions
        // s0 .. s0 + np - 1, contiguous) are read by gatherer gi as words
        // (2 k2 + gi) 32 + lane, k2 < kGatherWords; the stale ones are re-read
        // until all carry this launch's tag, and go to shared memory as they
        // are (the compute warps unpack their blocks).  A lane arrives on an expert's
        // barrier once its words of that expert are in (its k2 in
        // [klo(e), klo(e + 1))); every lane arrives for every expert, also when
        // a wait ran out, so that no compute warp waits on.
        const uint32_t want = a.stall_h ? 0x100u : (epoch & 0xFFu);  // (stall_h: a tag no CTA writes)
        const int gi = warp - kGather, nwe = FB * kHWords;
        const int P = max(1, 64 * kGatherWords / nwe);  // (nwe <= 64 kGatherWords: I <= kMaxI)
        auto klo = [&](int e) { return min(kGatherWords, max(0, (e * nwe - 32 * gi - lane + 63) / 64)); };
        bool ok = true;
        for (int s0 = 0; s0 < mp; s0 += P) {
            const int np = min(P, mp - s0), nf = np * nwe;
            const unsigned long long* src = a.hw + (size_t)s0 * nwe;
            unsigned long long* dst = hraw + (size_t)s0 * nwe;
            uint32_t todo = 0, left = (1u << np) - 1u;
#pragma unroll
            for (int k2 = 0; k2 < kGatherWords; ++k2)
                if ((2 * k2 + gi) * 32 + lane < nf) todo |= 1u << k2;
            const uint64_t t0 = globaltimer();
            while (true) {
                for (int e = 0; e < np; ++e) {
                    const uint32_t em = (1u << klo(e + 1)) - (1u << klo(e));
                    if (((left >> e) & 1u) && (!ok || !(todo & em))) {
                        mbar_arrive(hrdy0 + 8u * (s0 + e));
                        left &= ~(1u << e);
                        if (lane == 0 && gi == 0) {
                            trace_event(a, 208 + s0 + e);
                            if (s0 + e == 0) stamp(a, 3);
                        }
                    }
                }
                if (!todo || !ok) break;
                unsigned long long v[kGatherWords];
#pragma unroll
                for (int k2 = 0; k2 < kGatherWords; ++k2)
                    if ((todo >> k2) & 1u) v[k2] = ld_tagged(src + (2 * k2 + gi) * 32 + lane);
#pragma unroll
                for (int k2 = 0; k2 < kGatherWords; ++k2) {
                    if (((todo >> k2) & 1u) && (uint32_t)(v[k2] >> 56) == want) {
                        dst[(2 * k2 + gi) * 32 + lane] = v[k2];
                        todo &= ~(1u << k2);
                    }
                }
                if (todo && (globaltimer() - t0 > a.wait_ns || *abort_flag)) ok = false;
            }
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    raise_flag(a.err, ERR_TIMEOUT);
                }
                for (int sp = s0 + np; sp < mp; ++sp) mbar_arrive(hrdy0 + 8u * sp);
                break;
            }
        }
    } else if (warp < kComputeWarps) {
        // ------------------------------------------------------ compute warps
        // In every stage this warp takes K segment q = warp % NQx and the 4
        // consecutive rows 4 g .. 4 g + 3, g = warp / NQx (NQx = NQ or NQd
        // segments per row): lane l reads one 16-byte block of codes of each
        // row, and the slot goes back to the producer as soon as they are in
        // registers.  A down stage's 4-row runs each belong to one expert (d
        // is a multiple of 4).  After warp_sum4 lane 8 t holds row t's sum.
        const int t4 = 2 * ((lane >> 4) & 1) + ((lane >> 3) & 1);
        const bool writer = (lane & 7) == 0;
        const int nt = (a.I / 128) * (a.H / 128);  // tiles of a shared-expert matrix
        int slot = 0;
        uint32_t par = 0;
        bool ok = true;
        {
            // gate/up: block j's rows row0 .. row0 + RG (gate rows 0 .. 31,
            // up rows 32 .. 63 of the block) per stage, the token as operand
            const int rowb = a.H / 2, scb = a.H / kSB, g = warp / NQ;
            const uint8_t* wb = smem + Lo.ring + kRun * g * rowb + qx * 512 + lane * 16;
            const uint8_t* sb = smem + Lo.ring + kStageCodes + kRun * g * scb + (qx * 32 + lane) * (32 / kSB);
            float* pw = pgu + qx * 64 + kRun * g + t4;
            int row0 = 0, j = 0;  // h block j of this CTA, its rows row0 .. in the current stage
            for (int i = 0; i < p.ngur; ++i) {
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8u * slot, par, a.wait_ns, abort_flag));
                if (!ok) break;
                const uint8_t* w = wb + slot * kStageBytes;
                const uint8_t* sp = sb + slot * kStageBytes;
                uint4 wv[kRun];
                uint32_t sv[kRun];
#pragma unroll
                for (int t = 0; t < kRun; ++t) {
                    wv[t] = *reinterpret_cast<const uint4*>(w + t * rowb);
                    sv[t] = kNv ? *reinterpret_cast<const uint16_t*>(sp + t * scb) : sp[t * scb];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8u * slot);
                float v[kRun];
#pragma unroll
                for (int t = 0; t < kRun; ++t) v[t] = scaled_block<kNv>(wv[t], op, sv[t]) * opsf;
                const float r = warp_sum4(v[0], v[1], v[2], v[3], lane);
                if (writer) pw[j * NQ * 64 + row0] = r;
                if (++slot == kStages) {
                    slot = 0;
                    par ^= 1u;
                }
                row0 += p.RG;
                if (row0 == 64) {
                    // the last stage of h block j: this warp's partials of it are in
                    __syncwarp();
                    if (lane == 0) mbar_arrive(blk0 + 8u * j);
                    row0 = 0;
                    ++j;
                }
            }
        }
        if (kSh && ok && p.ngu > p.ngur) {
            // the shared expert's gate/up blocks: e4m3 rows of H bytes, RGs a
            // stage, this warp rows 2 g, 2 g + 1 (two 16-byte loads a row per
            // lane); one UE8M0 scale per 128 x 128 tile, in shared memory
            const int g = warp / NQ;
            const uint8_t* wb = smem + Lo.ring + kRunS * g * a.H + qx * 1024 + lane * 32;
            float* pw = pgu + qx * 64 + kRunS * g + t4;
            int row0 = 0, j = p.nbr;  // (the shared expert's blocks follow the routed ones)
            for (int i = p.ngur; i < p.ngu; ++i) {
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8u * slot, par, a.wait_ns, abort_flag));
                if (!ok) break;
                const uint8_t* w = wb + slot * kStageBytes;
                const uint4 w00 = *reinterpret_cast<const uint4*>(w), w01 = *reinterpret_cast<const uint4*>(w + 16);
                const uint4 w10 = *reinterpret_cast<const uint4*>(w + a.H);
                const uint4 w11 = *reinterpret_cast<const uint4*>(w + a.H + 16);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8u * slot);
                const int f = 32 * (c + j * G - m * FB);  // the block's first feature
                const float sc = ue8m0_to_f32(shs[(row0 < 32 ? 0 : nt) + (f >> 7) * (a.H / 128) + qx * 8 + (lane >> 2)]);
                const float v0 = block_dot_fp8(w00, w01, op) * sc * opsf;
                const float v1 = block_dot_fp8(w10, w11, op) * sc * opsf;
                const float r = warp_sum4(v0, v1, 0.f, 0.f, lane);
                if (writer && t4 < kRunS) pw[j * NQ * 64 + row0] = r;
                if (++slot == kStages) {
                    slot = 0;
                    par ^= 1u;
                }
                row0 += p.RGs;
                if (row0 == 64) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(blk0 + 8u * j);
                    row0 = 0;
                    ++j;
                }
            }
        }
        if (ok) {
            // down: the CTA's (kept expert s, row o) pairs as the flat list
            // u = s d + o, RD a stage; the warp's run starts at u, the operand
            // is expert s's h (K segment qh), switched when s changes
            const int rowb = a.I / 2, scb = a.I / kSB, g = warp / NQd, md = m * p.d;
            const uint8_t* wb = smem + Lo.ring + kRun * g * rowb + qh * 512 + lane * 16;
            const uint8_t* sb = smem + Lo.ring + kStageCodes + kRun * g * scb + (qh * 32 + lane) * (32 / kSB);
            int u = kRun * g, s = 0, sbase = 0, cur = -1;
            for (int i = p.ngu; i < p.ndr; ++i, u += p.RD) {
                const bool live = u < md;
                if (live) {
                    while (u >= sbase + p.d) {
                        sbase += p.d;
                        ++s;
                    }
                    if (s != cur) {
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(hrdy0 + 8u * s, 0, a.wait_ns, abort_flag));
                        if (!ok || *abort_flag) {
                            ok = false;
                            break;
                        }
                        load_h(hraw + ((size_t)s * FB + qh * 32 + lane) * kHWords, op, opsf);
                        cur = s;
                    }
                }
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8u * slot, par, a.wait_ns, abort_flag));
                if (!ok) break;
                const uint8_t* w = wb + slot * kStageBytes;
                const uint8_t* sp = sb + slot * kStageBytes;
                uint4 wv[kRun];
                uint32_t sv[kRun];
#pragma unroll
                for (int t = 0; t < kRun; ++t) {
                    wv[t] = *reinterpret_cast<const uint4*>(w + t * rowb);
                    sv[t] = kNv ? *reinterpret_cast<const uint16_t*>(sp + t * scb) : sp[t * scb];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8u * slot);
                if (live) {
                    float v[kRun];
#pragma unroll
                    for (int t = 0; t < kRun; ++t) v[t] = scaled_block<kNv>(wv[t], op, sv[t]) * opsf;
                    const float r = warp_sum4(v[0], v[1], v[2], v[3], lane);
                    if (writer) pdn[(s * NQd + qh) * a.dmax + (u - sbase) + t4] = r;
                }
                if (++slot == kStages) {
                    slot = 0;
                    par ^= 1u;
                }
            }
        }
        if (kSh && ok && p.n > p.ndr) {
            // the shared expert's down rows: e4m3 rows of I bytes, RDs a stage
            // (this warp rows u, u + 1 of the CTA's range), h of position m
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(hrdy0 + 8u * m, 0, a.wait_ns, abort_flag));
            if (ok && *abort_flag) ok = false;
            if (ok) load_h(hraw + ((size_t)m * FB + qh * 32 + lane) * kHWords, op, opsf);
            const int g = warp / NQd;
            const uint8_t* wb = smem + Lo.ring + kRunS * g * a.I + qh * 1024 + lane * 32;
            int u = kRunS * g;
            for (int i = p.ndr; ok && i < p.n; ++i, u += p.RDs) {
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8u * slot, par, a.wait_ns, abort_flag));
                if (!ok) break;
                const uint8_t* w = wb + slot * kStageBytes;
                const uint4 w00 = *reinterpret_cast<const uint4*>(w), w01 = *reinterpret_cast<const uint4*>(w + 16);
                const uint4 w10 = *reinterpret_cast<const uint4*>(w + a.I);
                const uint4 w11 = *reinterpret_cast<const uint4*>(w + a.I + 16);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8u * slot);
                if (u < p.d) {  // (rows u, u + 1: d is even; one 128-row tile, u and r0 being even)
                    const int row = p.r0 + u;
                    const float sc = ue8m0_to_f32(shs[2 * nt + (row >> 7) * (a.I / 128) + qh * 8 + (lane >> 2)]);
                    const float v0 = block_dot_fp8(w00, w01, op) * sc * opsf;
                    const float v1 = block_dot_fp8(w10, w11, op) * sc * opsf;
                    const float r = warp_sum4(v0, v1, 0.f, 0.f, lane);
                    if (writer && t4 < kRunS) pdn[(m * NQd + qh) * a.dmax + u + t4] = r;
                }
                if (++slot == kStages) {
                    slot = 0;
                    par ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            raise_flag(a.err, ERR_TIMEOUT);
        }
    }
    __syncthreads();
    stamp(a, 5);
    // the next launch of this CTA reads its count after this grid completed
    if (threadIdx.x == 0) a.launches[c] = epoch;
    if (*abort_flag) {
        tc::spin_ns(200000);  // (copies of a CTA that gave up land before it exits)
        return;
    }
    // ---- the combine of this CTA's rows: out[o] = sum over the kept experts
    // (ascending) of w_s * (its K segments' partials, in order)
    for (int i = threadIdx.x; i < p.d; i += kThreads) {
        float o = 0.f;
        for (int s = 0; s < m; ++s) {
            float y = 0.f;
            for (int q = 0; q < NQd; ++q) y += pdn[(s * NQd + q) * a.dmax + i];
            if (kNv) y *= __ldg(a.down_g + seg_e[s]);  // the matrix scale of the finished dot product
            o += seg_w[s] * y;
        }
        if (kSh) {  // the shared expert, unweighted, last
            float y = 0.f;
            for (int q = 0; q < NQd; ++q) y += pdn[(m * NQd + q) * a.dmax + i];
            o += y;
        }
        a.out[p.r0 + i] = o;
    }
}

// ------------------------------------------------------------------- host --
void split_table(int G, int m, int H, int I, bool nv, bool sh, int* cut) { split_rows(G, m, H, I, nv, sh, cut); }

bool supported(const moe_layer* L) {
    const moe_config& c = L->cfg;
    return (c.weight_format == MOE_WEIGHTS_MXFP4 || c.weight_format == MOE_WEIGHTS_NVFP4) && c.top_k <= kMaxK &&
           c.n_experts <= 1024 && L->gv_smem > 0;
}

// The down-row cuts of every kept count 1 .. k ([k][G + 1]), the largest h-block
// count and down range of a CTA over them, and the shared memory they need
// (0: more than a CTA has).
int smem_bytes(const moe_config& c, int G, int32_t* tab, int* nbmax, int* dmax) {
    const int FB = c.inter / 32, sh = c.has_shared ? 1 : 0;
    const bool nv = c.weight_format == MOE_WEIGHTS_NVFP4;
    *nbmax = ((c.top_k + sh) * FB + G - 1) / G;
    *dmax = 4;
    for (int m = 1; m <= c.top_k; ++m) {
        int32_t* cut = tab + (size_t)(m - 1) * (G + 1);
        split_rows(G, m, c.hidden, c.inter, nv, sh != 0, cut);
        for (int x = 0; x < G; ++x)
            if (cut[x + 1] - cut[x] > *dmax) *dmax = cut[x + 1] - cut[x];
    }
    const Layout Lo(c.hidden, c.inter, *nbmax, *dmax, nv, sh != 0);
    return Lo.total <= 227 * 1024 ? Lo.total : 0;
}

static const void* kernel_for(bool nv, bool sh) {
    return nv ? (sh ? reinterpret_cast<const void*>(k_decode_gemv<true, true>)
                    : reinterpret_cast<const void*>(k_decode_gemv<true, false>))
              : (sh ? reinterpret_cast<const void*>(k_decode_gemv<false, true>)
                    : reinterpret_cast<const void*>(k_decode_gemv<false, false>));
}

cudaError_t init(moe_layer* L) {
    L->gv_smem = 0;
    const moe_config& c = L->cfg;
    // K segments of 1024 elements dividing the 16 compute warps; a stage of
    // 32 KB of codes holds whole rows, a gate/up stage within one 32-row half
    // of a block (H >= 2048)
    if (c.hidden % kSeg || c.inter % kSeg || c.inter > kMaxI || c.hidden < 2 * kSeg ||
        kComputeWarps % (c.hidden / kSeg) || kComputeWarps % (c.inter / kSeg))
        return cudaSuccess;
    const int G = L->num_sms;
    int32_t* tab = new (std::nothrow) int32_t[(size_t)c.top_k * (G + 1)];
    if (!tab) return cudaErrorMemoryAllocation;
    int nbmax = 0, dmax = 0;
    const int bytes = smem_bytes(c, G, tab, &nbmax, &dmax);
    if (bytes == 0) {
        delete[] tab;
        return cudaSuccess;
    }
    const bool nv = c.weight_format == MOE_WEIGHTS_NVFP4;
    const void* kern = kernel_for(nv, c.has_shared != 0);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    int per_sm = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, bytes);
    if (e != cudaSuccess || per_sm < 1) {
        delete[] tab;
        return e;
    }
    // the down-row cuts of every kept count 1 .. k (the same on every call)
    e = cudaMalloc(&L->gv_rows, (size_t)c.top_k * (G + 1) * sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMemcpy(L->gv_rows, tab, (size_t)c.top_k * (G + 1) * sizeof(int32_t), cudaMemcpyHostToDevice);
    delete[] tab;
    if (e != cudaSuccess) return e;
    L->gv_smem = bytes;
    L->gv_nbmax = nbmax;
    L->gv_dmax = dmax;
    return cudaSuccess;
}

cudaError_t launch(moe_layer* L, const float* logits, const uint16_t* x, int32_t* ids, float* w, float* out,
                   cudaStream_t s, bool x_in_host) {
    Args a{};
    a.logits = logits;
    a.x = x;
    a.E = L->cfg.n_experts;
    a.k = L->cfg.top_k;
    a.H = L->cfg.hidden;
    a.I = L->cfg.inter;
    a.w_scale = L->cfg.w_scale;
    a.prune = RoutePrune{L->prune_keep, L->prune_min_w, L->prune_rho};
    a.ids_out = ids;
    a.w_out = w;
    a.out = out;
    a.gu_q = L->gu_q;
    a.gate_s = L->gate_s;
    a.up_s = L->up_s;
    a.down_q = L->down_q;
    a.down_s = L->down_s;
    a.gate_g = L->gate_g;
    a.up_g = L->up_g;
    a.down_g = L->down_g;
    a.sh = L->cfg.has_shared ? 1 : 0;
    a.sh_gu_q = L->sh_gu_q;
    a.sh_gate_s = L->sh_gate_s;
    a.sh_up_s = L->sh_up_s;
    a.sh_down_q = L->sh_down_q;
    a.sh_down_s = L->sh_down_s;
    a.hw = reinterpret_cast<unsigned long long*>(L->gv_words + gv_hword_off(L->num_sms));
    a.launches = L->gv_words + kGvCountOff;
    a.x_flag = L->gv_words + 2;
    a.x_stage = x_in_host ? L->x_stage : nullptr;
    a.err = L->d_err;
    a.wait_ns = L->wait_ns;
    a.stall_h = L->stall_next_decode;
    L->stall_next_decode = 0;  // one-shot
    a.nbmax = L->gv_nbmax;
    a.dmax = L->gv_dmax;
    a.RG = kStageCodes / (a.H / 2);
    a.RD = kStageCodes / (a.I / 2);
    a.spb = 64 / a.RG;
    a.RGs = kStageCodes / a.H;
    a.RDs = kStageCodes / a.I;
    a.spbs = 64 / a.RGs;
    a.rows = L->gv_rows;
    a.trace = L->trace;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L->num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L->gv_smem;
    cfg.stream = s;
    // cooperative (every CTA resident: they wait on each other's h flags) and
    // programmatic dependent launch (the prologue overlaps the previous kernel)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    L->launches += 1;
    const bool nv = L->cfg.weight_format == MOE_WEIGHTS_NVFP4, sh = L->cfg.has_shared != 0;
    return nv ? (sh ? cudaLaunchKernelEx(&cfg, k_decode_gemv<true, true>, a)
                    : cudaLaunchKernelEx(&cfg, k_decode_gemv<true, false>, a))
              : (sh ? cudaLaunchKernelEx(&cfg, k_decode_gemv<false, true>, a)
                    : cudaLaunchKernelEx(&cfg, k_decode_gemv<false, false>, a));
}

}  // namespace gemv
}  // namespace moe
