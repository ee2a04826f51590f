/*
 * moe.h -- C ABI of libmoe: the routed-expert FFN layer of a
 * DeepSeek-V4-Flash-style MoE on one NVIDIA GB300 (sm_103a).
 *
 * The layer ("DeepSeek-V4-Flash 284B - Deep-Dive Mathematical & Kernel
 * Guide", section 3.2, the FFN output equation):
 *     out(x) = shared(x) + sum_{i=1..k} w_i * expert_{e_i}(x),  sum_i w_i = w_scale
 * with expert(x) = W_down h, h_j = SiLU(g_j) * u_j, g = W_gate x, u = W_up x
 * (same guide, section 4).  Routed experts ship as MXFP4 (colibri "DeepSeek
 * V4 target engine", intro: "routed experts stay native fp4"): e2m1 codes in
 * 32-element blocks along the contraction axis, two codes per byte with the
 * even element in the low nibble, one UE8M0 scale byte 2^(c-127) per block.
 * The optional shared expert ships as fp8 e4m3 with one UE8M0 scale per
 * 128x128 tile (same page: "the dense set stays fp8-e4m3 with UE8M0 block
 * scales").  Activations enter every matmul as MXFP8: e4m3 codes in
 * 32-element blocks with a UE8M0 scale 2^(floor(log2 amax) - 8), rounded to
 * nearest even, saturating at +-448 (colibri "Linux CUDA tier": the MXFP8
 * tensor-core path).
 *
 * Conventions for every entry point:
 *  - All tensors are dense and row-major.  Pointers marked "device" must be
 *    device memory of the layer's GPU; "host" pointers are host memory (page-
 *    locked for the copies to overlap).  The caller owns every buffer it
 *    passes; the library never frees or keeps a caller pointer past the call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous: outputs are ready when the stream reaches
 *    that point.  route/permute/quantize/forward make no allocation and no
 *    host synchronisation, so they may be captured in a CUDA graph.
 *  - A layer is not thread-safe: calls on one layer must be serialised, and
 *    calls that overlap on the GPU (different streams) race on its workspace.
 *  - Every call returns a status and never aborts.  Invalid arguments that
 *    the host can see are rejected before anything is enqueued
 *    (MOE_ERR_INVALID_ARG).  Device-side checks (expert ids outside [0, E),
 *    token ids outside [0, V), a capped device wait that ran out) cannot be
 *    seen without a synchronisation: the kernels skip the offending work and
 *    raise a sticky device flag that moe_check() reports.  CUDA launch or
 *    runtime errors return MOE_ERR_CUDA.  moe_last_error() gives a message.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* bad pointer, size or id                      */
    MOE_ERR_UNSUPPORTED = 2, /* shape the kernels do not cover               */
    MOE_ERR_OOM = 3,         /* device allocation failed (create only)       */
    MOE_ERR_CUDA = 4,        /* CUDA runtime / launch error                  */
    MOE_ERR_TIMEOUT = 5      /* a capped device-side wait ran out            */
} moe_status;

/* Shape of one layer.  hidden (H) must be a multiple of 256 and inter (I) of
 * 128, both at most 8192;
 * 1 <= top_k (k) <= min(n_experts, 8); 1 <= n_experts (E) <= 1024;
 * max_tokens bounds T of every later call and sizes the workspace.  The
 * guide's layer (section 1): H = 4096, I = 2048, E = 256, k = 6,
 * w_scale = 1.5, one shared expert.                                        */
typedef struct {
    int hidden;
    int inter;
    int n_experts;
    int top_k;
    int max_tokens;
    int has_shared;  /* 1: the shared-expert pointers of moe_weights are set */
    float w_scale;   /* routing weights of a token sum to w_scale            */
    int weight_format; /* routed experts: MOE_WEIGHTS_MXFP4 (0, the default)
                        * or MOE_WEIGHTS_NVFP4 (1), see moe_weights         */
} moe_config;

/* Routed-expert weight formats.  MXFP4 is what the experts ship in (colibri
 * "DeepSeek V4 target engine", intro).  NVFP4-style (CISM VALIDATION,
 * "4-bit quantization scheme study", row "E2M1 + E4M3 b16 (NVFP4
 * granularity)", the best 4-bit scheme of that study): the same e2m1 codes,
 * one e4m3 scale per 16 elements along K and one fp32 scale per expert
 * matrix, element = e2m1 * e4m3 scale * matrix scale.  The tcgen05
 * block-scaled MMAs take UE8M0 scales per 32 elements only, so an NVFP4
 * layer runs its GEMMs on the CUDA cores (moe_set_gemm_path 2 returns
 * MOE_ERR_UNSUPPORTED); a one-token call takes the CUDA-core whole-layer
 * decode kernel where its shape rules hold (moe_set_decode_kernel), else
 * the grouped CUDA-core path.                                              */
enum { MOE_WEIGHTS_MXFP4 = 0, MOE_WEIGHTS_NVFP4 = 1 };

/* Device pointers to the weights, in the canonical shipping layout:
 *   gate_q, up_q  u8 [E][I][H/2]  e2m1 pairs (even element = low nibble)
 *   gate_s, up_s  u8 [E][I][H/32] UE8M0 block scales
 *                 (NVFP4: u8 [E][I][H/16] e4m3 block scales, positive)
 *   down_q        u8 [E][H][I/2]
 *   down_s        u8 [E][H][I/32] (NVFP4: [E][H][I/16] e4m3)
 *   gate_g, up_g, down_g  f32 [E]: NVFP4 only, the per-matrix scales
 *                 (ignored, may be NULL, for MXFP4)
 *   sh_gate_q, sh_up_q u8 [I][H] e4m3;  sh_gate_s, sh_up_s u8 [I/128][H/128]
 *   sh_down_q     u8 [H][I] e4m3;       sh_down_s          u8 [H/128][I/128]
 * Shared-expert pointers are ignored unless has_shared.                     */
typedef struct {
    const uint8_t *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
    const uint8_t *sh_gate_q, *sh_gate_s, *sh_up_q, *sh_up_s, *sh_down_q, *sh_down_s;
    const float *gate_g, *up_g, *down_g;
} moe_weights;

typedef struct moe_layer moe_layer;

/* Build a layer on the current CUDA device.  Copies and repacks the weights
 * into library-owned device memory (about 3.5 GB for the guide's shape) and
 * allocates the workspace for max_tokens; synchronises `stream` once, after
 * which the caller may free its weight buffers.  *out receives the layer, or
 * NULL on failure.                                                          */
moe_status moe_create(const moe_config* cfg, const moe_weights* w, moe_stream_t stream,
                      moe_layer** out);

/* Free everything the layer owns.  The caller must make sure no work of the
 * layer is still running (synchronise its streams first).  NULL is a no-op.*/
moe_status moe_destroy(moe_layer* layer);

/* Learned router (guide, section 1: gating_func = SQRT_SOFTPLUS, top-k over
 * the routed experts; section 3.2: the k weights sum to w_scale).
 *   logits  device f32 [T][E]
 *   ids     device i32 [T][k]  experts by descending score s = sqrt(softplus
 *           (logit)); equal scores go to the lower expert index
 *   w       device f32 [T][k]  w_j = w_scale * s_j / sum of the k scores
 * 1 <= T <= max_tokens.  The top-k is plain (one expert group).  With tail
 * pruning set (moe_set_route_prune) the pruned slots of a token come last
 * with id -1 and weight 0, and the kept weights are rescaled.  A token with
 * no valid selection (e.g. NaN logits) gets ids -1 and raises the device
 * flag.                                                                     */
moe_status moe_route(moe_layer* layer, const float* logits, int T, int32_t* ids, float* w,
                     moe_stream_t stream);

/* Hash router of the first layers (guide, section 1: ffn_gate_tid2eid maps a
 * token id to its experts; weights flat):
 *   token_ids device i32 [T] in [0, V); tid2eid device i32 [V][k]
 *   ids[t][j] = tid2eid[token_ids[t]][j];  w[t][j] = w_scale / k.
 * A token id outside [0, V) yields ids = -1 for that token and raises the
 * device flag (MOE_ERR_INVALID_ARG from moe_check).                         */
moe_status moe_route_hash(moe_layer* layer, const int32_t* token_ids, const int32_t* tid2eid,
                          int V, int T, int32_t* ids, float* w, moe_stream_t stream);

/* Token -> expert grouping (the grouping MUL_MAT_ID does; guide, section 2):
 * a stable counting sort of the rows r = t*k + j by expert ids[r].
 *   ids      device i32 [T][k], values in [0, E), or -1 for an empty slot
 *   offsets  device i32 [E+1]  offsets[e] = rows with expert < e
 *   row_src  device i32 [T*k]  row placed at sorted position p (ascending r
 *            within an expert's segment); entries past offsets[E] unused
 *   row_dst  device i32 [T*k]  inverse: sorted position of row r
 * An id of -1 (a pruned expert) is left out quietly (row_dst = -1); other
 * ids outside [0, E) are left out and raise the device flag.               */
moe_status moe_permute(moe_layer* layer, const int32_t* ids, int T, int32_t* offsets,
                       int32_t* row_src, int32_t* row_dst, moe_stream_t stream);

/* Activation quantiser, exposed for tests: bf16 rows -> MXFP8.
 *   x  device u16 [T][H] (bf16 bits);  q device u8 [T][H] e4m3 codes;
 *   s  device u8 [T][H/32] UE8M0 byte of 2^(floor(log2 amax) - 8) per
 *      32-block (amax = 0 or a clamped exponent gives -127 -> byte 0).     */
moe_status moe_quantize(moe_layer* layer, const uint16_t* x, int T, uint8_t* q, uint8_t* s,
                        moe_stream_t stream);

/* The layer: permute, quantise, SwiGLU gate/up with MXFP8 requantisation of
 * h, down projection, and the weighted combine in ascending expert order,
 * plus the shared expert when present.
 *   x    device u16 [T][H] bf16;  ids device i32 [T][k] in [0, E), or -1
 *        for an empty slot, which adds nothing;
 *   w    device f32 [T][k];       out device f32 [T][H] (overwritten).     */
moe_status moe_forward(moe_layer* layer, const uint16_t* x, int T, const int32_t* ids,
                       const float* w, float* out, moe_stream_t stream);

/* Routing and layer in one call: moe_route followed by moe_forward, with
 * ids [T][k] and w [T][k] (device) written as moe_route writes them and out
 * [T][H] as moe_forward.  Small batches (T <= 32) run the routing, the
 * counting sort and the quantisation in one kernel.  One token on the
 * automatic path runs as one cooperative kernel of one CTA per SM (route,
 * quantise, gate/up, down, combine; hand-offs between CTAs through bounded
 * waits on flags or on epoch-tagged data); moe_hidden does not report h
 * after such a call.                                                       */
moe_status moe_route_forward(moe_layer* layer, const float* logits, const uint16_t* x, int T,
                             int32_t* ids, float* w, float* out, moe_stream_t stream);

/* Whole layer from host memory: copies x (host u16 [T][H]) and logits (host
 * f32 [T][E]) into the layer's staging buffers, runs moe_route and
 * moe_forward, and copies the result to out (host f32 [T][H]).  Asynchronous
 * on `stream` (page-locked host buffers make the copies overlap); read out
 * only after synchronising the stream.  One token on the automatic path with
 * all three buffers page-locked (16-byte aligned x and out) enqueues no copy:
 * the decode kernel reads and writes the host memory in place (mapped; one
 * CTA reads x over the host link and hands a device copy to the others).   */
moe_status moe_forward_host(moe_layer* layer, const uint16_t* x, const float* logits, int T,
                            float* out, moe_stream_t stream);

/* Test hook: after moe_forward, the requantised SwiGLU activations of the
 * rows r = t*k + j of its T tokens, in row order:
 *   hq device u8 [T*k][I] e4m3;  hs device u8 [T*k][I/32] UE8M0.          */
moe_status moe_hidden(moe_layer* layer, int T, uint8_t* hq, uint8_t* hs, moe_stream_t stream);

/* Synchronise `stream` and report (then clear) the sticky device flag:
 * MOE_OK, MOE_ERR_INVALID_ARG (an id was out of range) or MOE_ERR_TIMEOUT. */
moe_status moe_check(moe_layer* layer, moe_stream_t stream);

/* Bytes of device workspace moe_create allocates for this shape (weights
 * not included); 0 for an invalid configuration.                           */
size_t moe_workspace_bytes(const moe_config* cfg);

/* Message of the last failed call on `layer`; for layer == NULL, of the last
 * failed call in this thread that had no layer (e.g. moe_create).          */
const char* moe_last_error(const moe_layer* layer);

/* Stage timing: when `events` is non-NULL, the next moe_forward call on
 * `layer` records events[0..5] on its stream at the stage boundaries
 * [start, after permute, after quantise, after gate/up, after down (and the
 * shared expert), after combine] and then forgets the array.  events holds
 * 6 cudaEvent_t created by the caller; n must be 6.  Recording is stream-
 * ordered, so it may be captured in a CUDA graph.                         */
moe_status moe_set_stage_events(moe_layer* layer, void* const* events, int n);

/* Kernel trace (diagnostics): when `buf` is non-NULL, the next moe_forward /
 * moe_route_forward on `layer` records global-timer values and wait times in
 * buf (device u64): tensor-core GEMM launch j (0 gate/up, 1 down, 2 and 3 the
 * shared expert) writes 12 counters per CTA at buf + (j * num_sms + cta) * 12:
 * [entry ns, exit ns, producer ns waiting for free stages, MMA ns waiting for
 * data, MMA ns waiting for the accumulator, epilogue ns waiting for the
 * accumulator, epilogue ns working, K-stages issued, ns when the wait for the
 * previous kernel ended]; the one-CTA front kernel of small batches writes
 * [entry, wait end, exit] at buf + 4 * num_sms * 12; the CUDA-core decode
 * kernel writes per CTA [entry, -, publisher done, first h gathered, first
 * copy issued, final barrier] ns at buf + 8 * cta and, for CTAs 0, 1, 80 and
 * num_sms - 1 (t = 0 .. 3), event times at buf + 8 * num_sms + 256 * t + i
 * (i = 128 + stage: copy issued; 192 + j, 200 + j: h block j computed,
 * published; 208 + s: kept expert s's h gathered).  entries >=
 * max(48 * num_sms + 4, 8 * num_sms + 1024), else MOE_ERR_INVALID_ARG.
 * One-shot, like moe_set_stage_events.                                    */
moe_status moe_set_trace(moe_layer* layer, unsigned long long* buf, size_t entries);

/* Number of CUDA kernels this layer has enqueued since moe_create (a launch
 * made while a stream is being captured counts once, although every replay
 * of the graph runs it again).                                             */
unsigned long long moe_kernel_launches(const moe_layer* layer);

/* Kernel path of the GEMM steps: 0 = automatic (tcgen05 when the device is
 * sm_103, and a one-token moe_route_forward / moe_forward_host as a single
 * whole-layer decode kernel where the shape allows one: see
 * moe_set_decode_kernel), 1 = CUDA-core kernels, 2 = tcgen05 block-scaled
 * tensor-core kernels only (never a decode kernel).  All compute the same layer; the
 * choice only affects speed and the order of fp32 additions.               */
moe_status moe_set_gemm_path(moe_layer* layer, int path);

/* Which whole-layer kernel a one-token call on the automatic GEMM path
 * (moe_route_forward / moe_forward_host with T = 1) takes.  kind 0 =
 * automatic: the CUDA-core split-K GEMV kernel where the shape allows it
 * (MXFP4 or NVFP4 experts, H and I multiples of 1024 with H / 1024 and
 * I / 1024 dividing 16, H >= 2048, with or without the shared expert, and
 * its shared-memory layout -- a 5-stage weight ring, the h of the kept
 * experts (and the shared one), the CTA's partial sums -- within 227 KB:
 * e.g. I <= 2048 for top_k <= 8, not I = 4096 with 6 experts), else the
 * tcgen05 kernel (MXFP4, H <= 4096, I <= 2048, no shared expert), else the
 * grouped kernels; 1 = the CUDA-core kernel; 2 = the tcgen05 kernel.  Both
 * compute the layer for a
 * single decode token (guide, section 2.A: one token, the MUL_MAT_ID of its
 * top-k experts), with the combine in ascending expert order; they differ
 * only in the order of fp32 additions.
 * MOE_ERR_UNSUPPORTED if the layer's shape has no such kernel,
 * MOE_ERR_INVALID_ARG for another kind; the setting is then unchanged.
 * Not part of the method: a switch for benchmarks and tests.             */
moe_status moe_set_decode_kernel(moe_layer* layer, int kind);

/* The whole-layer kernel a one-token call of this layer takes with its
 * current settings: *kind = 0 none (the grouped kernels), 1 the CUDA-core
 * GEMV kernel, 2 the tcgen05 kernel (the codes of moe_set_decode_kernel).
 * A diagnostic for benchmarks and tests.                                  */
moe_status moe_decode_info(const moe_layer* layer, int* kind);

/* Tail pruning of the learned router (guide, section 3.2 item 3: top-k
 * below the layer's k and the adaptive tail, with L2-quadrature rescaling;
 * RFC on CPU kernels, item 5: dropping experts under a weight threshold).
 * Applies to moe_route, moe_route_forward and moe_forward_host from the
 * next call on; the hash router is never pruned.  Per token, in router
 * order: expert 0 is kept; expert j >= 1 while j < keep and w_j >= min_w
 * (the first that fails ends the kept prefix of m experts).  The kept
 * weights are multiplied by
 *   sqrt(((1 - rho) S2 + rho S1^2) / ((1 - rho) S2' + rho S1'^2)),
 * S1, S2 = sum of w and of w^2 over all k, S1', S2' over the kept experts:
 * rho = 0 keeps the sum of squares (orthogonal expert outputs), rho = 1
 * the sum (linear rescaling).  The pruned slots get id -1 and weight 0 and
 * their experts' weights are never read.
 *   1 <= keep (keep >= k: no count limit); min_w finite (<= 0: no
 *   threshold); 0 <= rho <= 1.  keep >= k with min_w <= 0 turns it off (the
 *   default).  MOE_ERR_INVALID_ARG otherwise, the setting unchanged.       */
moe_status moe_set_route_prune(moe_layer* layer, int keep, float min_w, float rho);

/* Wall-time limit of every device-side wait of this layer's kernels (a
 * pipeline barrier, or a flag or tagged word another CTA writes): a wait that
 * runs out gives up instead of spinning on.  The kernel then skips its
 * remaining work, lets its copies in flight land, frees its tensor memory and
 * exits; the device flag it raises makes the next moe_check() return
 * MOE_ERR_TIMEOUT (outputs of that call are undefined), and the layer stays
 * usable.  Not part of the method: a guard against a CTA that never arrives
 * (colibri "DeepSeek V4 target engine", "Validation": every GPU stage is
 * checked against the CPU, and a failure must surface, not hang).
 *   seconds in [1e-4, 60]; default 2.  MOE_ERR_INVALID_ARG otherwise.      */
moe_status moe_set_wait_limit(moe_layer* layer, double seconds);

/* Test hook of the bounded-wait path above.  The next one-token call that
 * runs the whole-layer decode kernel (moe_route_forward or moe_forward_host
 * with T = 1 on the automatic path) waits for its gate/up results under a
 * value no CTA ever writes, so every CTA's wait runs out after the wait
 * limit and the call ends with MOE_ERR_TIMEOUT at the next moe_check().
 * One-shot: the call after it runs normally.  MOE_ERR_UNSUPPORTED if the
 * layer has no decode kernel (shape, or not an sm_103 GPU).               */
moe_status moe_test_stall_next_decode(moe_layer* layer);

/* Host-side view of the CUDA-core decode kernel's work split, for tests (no
 * GPU needed): cut[x], x = 0 .. num_sms, receives the first output row of
 * CTA x of num_sms for `kept` kept experts of a layer with this hidden and
 * inter size, NVFP4 (nvfp4 != 0) or MXFP4 weights and a shared expert
 * (shared != 0) or none; CTA x owns rows [cut[x], cut[x + 1]) of every
 * expert.  The h blocks (kept * inter / 32 routed ones, then the shared
 * expert's inter / 32) go to CTA b mod num_sms; the rows are cut in
 * proportion to what each CTA has left of an equal share of the stream
 * bytes, every cut rounded to a multiple of 4.  cut (host, num_sms + 1
 * ints) is caller-owned.  MOE_ERR_INVALID_ARG for num_sms < 1, kept < 1,
 * hidden or inter not positive multiples of 1024 or above 8192, or a NULL
 * cut.                                                                     */
moe_status moe_test_decode_split(int num_sms, int kept, int hidden, int inter, int nvfp4, int shared,
                                 int* cut);

/* Token -> expert grouping without a layer and without any allocation.
 * The method's description has no counterpart: this entry point exists for callers that
 * cannot call cudaMalloc -- code running inside another framework's memory
 * arena that forbids foreign allocations, serving loops that freeze device
 * memory after start-up, or engines that only want the grouping for their
 * own expert GEMMs and cannot afford moe_create's weight copies.  It runs the
 * same stable counting sort as moe_permute and gives the same results:
 *   ids      device i32 [T][top_k];  offsets device i32 [n_experts+1];
 *   row_src, row_dst device i32 [T*top_k]  (as moe_permute).
 * Limits: 1 <= T*top_k <= 65536, 1 <= top_k <= 8, 1 <= n_experts <= 1024;
 * larger sizes return MOE_ERR_INVALID_ARG (message in moe_last_error(NULL)).
 * The sort's bookkeeping lives in one static device array of 1,060,876 bytes
 * that every GPU loading the library holds until the process exits; every
 * call shares it, so calls that overlap on the GPU (several streams or
 * threads at once) race and must be serialised by the caller.  The first
 * call on a device looks up that array's address and sets the kernel's
 * shared-memory limit (with the device current): make it before any stream
 * capture; later calls only enqueue one kernel and may be captured.  Ids
 * outside [0, n_experts) are left out (row_dst = -1); with no layer there is
 * no device flag to report them.                                           */
moe_status moe_permute_noalloc(const int32_t* ids, int T, int top_k, int n_experts,
                               int32_t* offsets, int32_t* row_src, int32_t* row_dst,
                               moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
