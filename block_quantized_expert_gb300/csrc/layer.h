// layer.h -- the moe_layer object behind the C ABI and the launchers of its
// kernels.  Everything here is library-internal.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/moe.h"

struct moe_layer {
    moe_config cfg;
    int device;
    int num_sms;
    int gemm_path;  // 0 auto, 1 CUDA cores, 2 tcgen05
    // tail pruning of the learned routing (keep = top_k, min_w = 0: none)
    int prune_keep;
    float prune_min_w, prune_rho;
    uint64_t wait_ns;        // wall-time limit of every device-side wait
    int stall_next_decode;   // test hook: the next decode launch's h waits cannot complete

    // -------- weights (library-owned copies) --------
    // gate/up codes interleaved per 128 features: [E][I/128][gate 128 rows, up 128 rows][H/2],
    // so one 256-row copy brings the gate and up tiles of 128 features; down codes canonical
    // [E][H][I/2]; scales canonical [E][rows][K/32] (NVFP4: e4m3 [E][rows][K/16]; read by the
    // CUDA-core kernels).
    uint8_t *gu_q, *gate_s, *up_s, *down_q, *down_s;
    float *gate_g, *up_g, *down_g;  // NVFP4: per-expert matrix scales [E] (null for MXFP4)
    uint8_t *sh_gu_q, *sh_gate_s, *sh_up_s, *sh_down_q, *sh_down_s;  // shared: [I/128][256][H] e4m3
    // scales as 512-byte atoms, two per 256-row block and 128-column step:
    // [blocks][K/128][2][512] (gate/up: gate, up halves; down: rows 0-127, 128-255)
    uint8_t *gu_sf, *down_sf, *sh_gu_sf, *sh_down_sf;

    // -------- workspace (sized by max_tokens) --------
    int R_max;        // max_tokens * k
    int Rp_max;       // padded permuted rows (segments start at multiples of 128)
    int32_t* counts;      // [E]   rows per expert
    int32_t* offsets;     // [E+1] unpadded segment starts
    int32_t* poff;        // [E+1] padded segment starts (multiples of 128)
    int32_t* tile_scan;   // [E+1] 128-row tiles before expert e
    int32_t* chunk_scan;  // [E+1] CUDA-core token chunks before expert e
    int32_t* row_src;     // [R]
    int32_t* row_dst;     // [R]
    int32_t* row_pos;     // [R]  padded position of row r (-1 if dropped)
    int32_t* pos_row;     // [Rp] row at padded position p (-1 = padding)
    int32_t* sh_desc;     // shared-expert segment: counts[1], poff[2], tiles[2], chunks[2]
    int32_t* perm_cnt;    // [R/1024 chunks][E] expert counts of the grid-wide sort
    uint8_t* xq;          // [Rp][H]   MXFP8 codes of x, permuted rows
    uint8_t* xs;          // atoms of [Rp][H/32]
    uint8_t* xq_tok;      // [T][H]    MXFP8 codes of x, token order (shared expert)
    uint8_t* xs_tok;      // atoms of [T_pad][H/32]
    uint8_t* hq;          // [Rp][I]   MXFP8 codes of h
    uint8_t* hs;          // atoms
    uint8_t* hq_sh;       // [T_pad][I] shared expert h
    uint8_t* hs_sh;
    float* y;             // [R][H]   down output of row r (unweighted)
    float* y_sh;          // [T][H]   shared expert output
    uint16_t* x_stage;    // [T][H]   moe_forward_host staging
    float* logits_stage;  // [T][E]
    float* out_stage;     // [T][H]
    int32_t* ids_stage;   // [T][k]
    float* w_stage;       // [T][k]
    uint32_t* d_err;      // sticky device error flags
    int32_t* sk_counters; // [4][num_sms] arrival counters of split tiles (zeroed per forward)
    float* sk_partials;   // [num_sms][2][2][128][128] partial accumulators of split tiles
    unsigned long long* dec_yw;  // [128 tiles][256] decode down outputs: launch epoch << 32 | fp32 bits
    // the CUDA-core decode kernel: its words (the staged-x flag, the h-block
    // flags [8][I/32], the CTAs' launch counts), its shared memory and work
    // bounds (gv_smem 0: the kernel is not available)
    uint32_t* gv_words;
    int32_t* gv_rows;  // its down-row cuts: [k][num_sms + 1] for each kept count 1 .. k
    int gv_smem, gv_nbmax, gv_dmax;
    int decode_kernel;  // one-token calls: 0 automatic, 1 the CUDA-core kernel, 2 the tcgen05 kernel

    void* tc;             // tensor-core kernel state (tensor maps), or null
    unsigned long long launches;  // kernels enqueued so far
    unsigned long long* trace;    // one-shot kernel trace buffer (diagnostics), or null
    cudaEvent_t stage_ev[6];  // one-shot stage events for the next forward
    int stage_ev_set;

    char last_error[256];
};

namespace moe {

constexpr int kChunk = 4;      // tokens per CUDA-core GEMM work item
constexpr int kFrontMaxT = 32; // batches up to this size use the one-CTA front kernel
// the combine fused into the down GEMM up to this size: the CTA that
// finishes a feature block combines it for every token, a tail that grows
// with T (at T = 32 a separate combine kernel is faster, measured)
constexpr int kFusedCombineMaxT = 4;
// the front kernel quantises x itself up to this size; larger batches
// quantise in a grid-wide kernel (one SM is instruction-bound on the
// scattered stores: about 1 us per token of T = 32, top-6, H = 4096)
constexpr int kFrontQuantMaxT = 4;

// split-tile counters of the grouped GEMMs (4 launches x num_sms, then one
// per 256-feature block of the fused combine, H / 256 <= 32): zeroed by every
// grouped forward
inline int kSkZeroed(const moe_layer* L) { return 4 * L->num_sms + 32; }
// then the words of the one-token decode kernel, zeroed only at creation: a
// 64-bit launch counter, piece flags [4 phases][num_sms][2], h flags [128],
// the staged-x flag (+ spare)
inline int kDecWords(const moe_layer* L) { return 2 + 8 * L->num_sms + 128 + 32; }
inline int kSkCounters(const moe_layer* L) { return kSkZeroed(L) + kDecWords(L); }

// 32-bit words of the CUDA-core decode kernel, zeroed at creation: spare
// [0, 2), staged-x flag [2], spare [3], the CTAs' launch counts [num_sms] from
// kGvCountOff, then (8-byte aligned) the published h: [9 positions: up to 8
// kept experts, then the shared expert][I/32 blocks][6] 64-bit tagged words
constexpr int kGvCountOff = 4;
inline size_t gv_hword_off(int num_sms) { return ((size_t)kGvCountOff + num_sms + 1) / 2 * 2; }
inline size_t gv_words_count(const moe_config& c, int num_sms) {
    return gv_hword_off(num_sms) + (size_t)2 * 9 * (c.inter / 32) * 6;
}

// Launch with a programmatic (early-launch) edge to the previous kernel of the
// stream; the kernels synchronise on it with pdl_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers; each returns the launch error (cudaSuccess on success).
cudaError_t launch_route(moe_layer* L, const float* logits, int T, int32_t* ids, float* w,
                         cudaStream_t s);
cudaError_t launch_route_hash(moe_layer* L, const int32_t* tok, const int32_t* tab, int V,
                              int T, int32_t* ids, float* w, cudaStream_t s);
// Counting sort into the given outputs plus the layer's padded bookkeeping.
cudaError_t launch_permute(moe_layer* L, const int32_t* ids, int T, int32_t* offsets,
                           int32_t* row_src, int32_t* row_dst, cudaStream_t s);
cudaError_t launch_quantize_canonical(moe_layer* L, const uint16_t* x, int T, uint8_t* q,
                                      uint8_t* sc, cudaStream_t s);
cudaError_t launch_quantize_scatter(moe_layer* L, const uint16_t* x, int T, cudaStream_t s);
// route (if logits) + permute (+ quantise, if x) in one CTA, for T <= kFrontMaxT
cudaError_t launch_front(moe_layer* L, const float* logits, int32_t* ids, float* w, const uint16_t* x,
                         int T, cudaStream_t s);
cudaError_t launch_combine(moe_layer* L, const int32_t* ids, const float* w, int T,
                           float* out, cudaStream_t s);
cudaError_t launch_hidden_gather(moe_layer* L, int T, uint8_t* hq, uint8_t* hs,
                                 cudaStream_t s);
cudaError_t launch_gemm_cc(moe_layer* L, int T, cudaStream_t s, cudaEvent_t mid);
cudaError_t launch_permute_raw(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                               int32_t* row_src, int32_t* row_dst, int32_t* counts, int32_t* poff,
                               int32_t* tile_scan, int32_t* chunk_scan, int32_t* row_pos,
                               int32_t* pos_row, cudaStream_t s);
cudaError_t kernels_init();
void set_thread_error(const char* msg);
cudaError_t cc_init();

// Tensor-core path.
cudaError_t tc_init(moe_layer* L);
bool decode_supported(const moe_layer* L);
// x_in_host: x is mapped host memory; one CTA copies it to the layer's
// staging buffer for the others (one read of x over the host link, not one
// per CTA)
cudaError_t launch_decode(moe_layer* L, const float* logits, const uint16_t* x, int32_t* ids, float* w,
                          float* out, cudaStream_t s, bool x_in_host = false);
void tc_free(moe_layer* L);

// The one-token layer as a split-K GEMV on the CUDA cores (decode_gemv.cu).
namespace gemv {
cudaError_t init(moe_layer* L);      // sets gv_smem / gv_nbmax / gv_dmax (0: not available)
bool supported(const moe_layer* L);  // shape, weight format, init succeeded
// rows [cut[x], cut[x + 1]) of CTA x of G for m kept experts (cut: G + 1 entries)
void split_table(int G, int m, int H, int I, bool nv, bool sh, int* cut);
cudaError_t launch(moe_layer* L, const float* logits, const uint16_t* x, int32_t* ids, float* w, float* out,
                   cudaStream_t s, bool x_in_host);
}  // namespace gemv
// cmb_ids != null: fuse the combine into the down GEMM (out = sum over the
// token's experts in ascending order of w * y); requires no shared expert.
cudaError_t launch_gemm_tc(moe_layer* L, int T, cudaStream_t s, cudaEvent_t mid, const int32_t* cmb_ids,
                           const float* cmb_w, float* cmb_out);
// Scale atoms of 256-row blocks (two 512-byte atoms per block and 128-column
// step).  mode 0: halves from srcA / srcB (block g rows g*128..), canonical
// [mats][rows][K/32] scales; 1: halves = rows (2g)*128.. and (2g+1)*128.. of srcA;
// 2 and 3: the same from 128x128 tile scales [rows/128][K/128] (mats = 1).
cudaError_t pack_sf_pairs(const uint8_t* srcA, const uint8_t* srcB, uint8_t* dst, int mats,
                          int groups, int K, int mode, cudaStream_t s);

}  // namespace moe
