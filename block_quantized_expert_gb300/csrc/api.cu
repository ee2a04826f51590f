// api.cu -- the C ABI of libmoe (include/moe.h): argument checks, the layer
// object and its workspace, and the sequence of kernels of one layer call.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <new>

#include "common.cuh"
#include "layer.h"
#include "stage_event.h"

namespace {

thread_local char g_tls_error[256] = "";

moe_status fail(moe_layer* L, moe_status st, const char* fmt, ...) {
    char* buf = L ? L->last_error : g_tls_error;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, 256, fmt, ap);
    va_end(ap);
    return st;
}

moe_status cuda_fail(moe_layer* L, cudaError_t e, const char* what) {
    return fail(L, MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Sizes {
    size_t R, Rp, Tpad;
};

Sizes sizes_of(const moe_config& c) {
    Sizes z;
    z.R = (size_t)c.max_tokens * c.top_k;
    size_t nz = z.R < (size_t)c.n_experts ? z.R : (size_t)c.n_experts;
    z.Rp = round_up(z.R + nz * (moe::kRowTile - 1), moe::kRowTile);
    z.Tpad = round_up((size_t)c.max_tokens, moe::kRowTile);
    return z;
}

// Device address of page-locked (mapped) host memory; false for device or
// pageable memory.
bool mapped_host(const void* p, const void** dp) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return false;
    *dp = at.devicePointer;
    return true;
}

const char* check_config(const moe_config* c) {
    if (!c) return "config is NULL";
    if (c->hidden <= 0 || c->hidden % 128) return "hidden must be a positive multiple of 128";
    if (c->inter <= 0 || c->inter % 128) return "inter must be a positive multiple of 128";
    if (c->n_experts < 1 || c->n_experts > moe::kMaxExperts) return "n_experts must be in [1, 1024]";
    if (c->top_k < 1 || c->top_k > moe::kMaxTopK || c->top_k > c->n_experts)
        return "top_k must be in [1, min(n_experts, 8)]";
    if (c->max_tokens < 1 || (long long)c->max_tokens * c->top_k > (1LL << 30))
        return "max_tokens out of range";
    if (c->hidden > 8192 || c->inter > 8192) return "hidden/inter larger than 8192";
    if (c->hidden % 256) return "hidden must be a multiple of 256";
    if (!std::isfinite(c->w_scale)) return "w_scale must be finite";
    if (c->weight_format != MOE_WEIGHTS_MXFP4 && c->weight_format != MOE_WEIGHTS_NVFP4)
        return "weight_format must be MOE_WEIGHTS_MXFP4 or MOE_WEIGHTS_NVFP4";
    return nullptr;
}

// Workspace byte count: every device buffer moe_create allocates besides the
// weight copies.
size_t workspace_bytes(const moe_config& c) {
    Sizes z = sizes_of(c);
    const size_t H = c.hidden, I = c.inter, E = c.n_experts, T = c.max_tokens, k = c.top_k;
    size_t b = 0;
    b += 5 * (E + 1) * 4;                        // counts, offsets, poff, tile_scan, chunk_scan
    b += 3 * z.R * 4 + z.Rp * 4 + 8 * 4;         // row_src, row_dst, row_pos, pos_row, sh_desc
    b += (z.R + 1023) / 1024 * E * 4;            // perm_cnt
    b += z.Rp * H + z.Rp * H / 32;               // xq, xs
    b += z.Rp * I + z.Rp * I / 32;               // hq, hs
    b += z.R * H * 4;                            // y
    if (c.has_shared) {
        b += z.Tpad * H + z.Tpad * H / 32 + z.Tpad * I + z.Tpad * I / 32 + T * H * 4;
    }
    b += T * H * 2 + T * E * 4 + T * H * 4 + 2 * T * k * 4;  // staging
    b += 256;                                    // error word
    // split-tile counters, decode flags and partial accumulators (sized for up to 256 SMs)
    b += (size_t)((4 * 256 + 32) + (2 + 8 * 256 + 128 + 32)) * 4 + (size_t)256 * 2 * 2 * 128 * 128 * 4;
    b += (size_t)128 * 256 * 8;                  // decode down outputs with their epoch
    b += (size_t)moe::gv_words_count(c, 256) * 4;  // CUDA-core decode kernel: flags, launch counts (<= 256 SMs)
    return b;
}

template <typename P>
cudaError_t dalloc(P** p, size_t bytes, size_t* total) {
    *total += bytes;
    return cudaMalloc((void**)p, bytes ? bytes : 1);
}

void free_all(moe_layer* L) {
    void* ptrs[] = {L->gu_q, L->gate_s, L->up_s, L->down_q, L->down_s,
                    L->sh_gu_q, L->sh_gate_s, L->sh_up_s, L->sh_down_q, L->sh_down_s,
                    L->gu_sf, L->down_sf, L->sh_gu_sf, L->sh_down_sf,
                    L->counts, L->offsets, L->poff, L->tile_scan, L->chunk_scan, L->row_src,
                    L->row_dst, L->row_pos, L->pos_row, L->sh_desc, L->perm_cnt, L->xq, L->xs, L->xq_tok,
                    L->xs_tok, L->hq, L->hs, L->hq_sh, L->hs_sh, L->y, L->y_sh, L->x_stage,
                    L->logits_stage, L->out_stage, L->ids_stage, L->w_stage, L->d_err,
                    L->sk_counters, L->sk_partials, L->dec_yw, L->gate_g, L->up_g, L->down_g,
                    L->gv_words, L->gv_rows};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    moe::tc_free(L);
}

moe_status check_T(moe_layer* L, int T) {
    if (T < 1 || T > L->cfg.max_tokens)
        return fail(L, MOE_ERR_INVALID_ARG, "T=%d outside [1, max_tokens=%d]", T, L->cfg.max_tokens);
    return MOE_OK;
}


}  // namespace

namespace moe {
void set_thread_error(const char* msg) { snprintf(g_tls_error, sizeof(g_tls_error), "%s", msg); }
}  // namespace moe

namespace {

// The whole-layer kernel a one-token call takes: 0 none (the grouped
// kernels), 1 the CUDA-core GEMV kernel, 2 the tcgen05 kernel.  Automatic:
// the CUDA-core kernel where its shape allows, else the tcgen05 one.
int decode_kind(const moe_layer* L) {
    if (L->gemm_path != 0) return 0;
    const bool gv = moe::gemv::supported(L), tcd = L->tc != nullptr && moe::decode_supported(L);
    if (L->decode_kernel == 1) return gv ? 1 : 0;
    if (L->decode_kernel == 2) return tcd ? 2 : 0;
    return gv ? 1 : (tcd ? 2 : 0);
}

cudaError_t launch_decode_kind(moe_layer* L, int kind, const float* logits, const uint16_t* x, int32_t* ids,
                               float* w, float* out, cudaStream_t s, bool x_in_host) {
    return kind == 1 ? moe::gemv::launch(L, logits, x, ids, w, out, s, x_in_host)
                     : moe::launch_decode(L, logits, x, ids, w, out, s, x_in_host);
}

// The kernels of one layer call.  Small batches (T <= kFrontMaxT) run the
// routing (when logits are given), the counting sort and the quantisation in
// one CTA; on the tensor-core path without a shared expert the combine is
// fused into the down GEMM.  `mark(i, e)` records stage event i (optional).
cudaError_t forward_kernels(moe_layer* L, const float* logits, const uint16_t* x, int T, int32_t* ids,
                            float* w, float* out, cudaStream_t s,
                            const std::function<cudaError_t(int, cudaError_t)>& mark) {
    auto M = [&](int i, cudaError_t e) { return mark ? mark(i, e) : e; };
    const bool small = T <= moe::kFrontMaxT;
    const bool tc = L->gemm_path != 1 && L->tc != nullptr;  // automatic: tensor cores
    const bool fuse_combine = tc && small && !L->cfg.has_shared && T <= moe::kFusedCombineMaxT;
    cudaError_t e = M(0, cudaSuccess);
    const int dk = logits && T == 1 ? decode_kind(L) : 0;
    if (dk) {
        // one token: the whole layer in one cooperative kernel (the stage
        // marks before it are empty and its time shows as the gate/up stage)
        if (e == cudaSuccess) e = M(1, cudaSuccess);
        if (e == cudaSuccess) e = M(2, cudaSuccess);
        if (e == cudaSuccess) e = launch_decode_kind(L, dk, logits, x, ids, w, out, s, false);
        if (e == cudaSuccess) e = M(3, cudaSuccess);
        if (e == cudaSuccess) e = M(4, cudaSuccess);
        if (e == cudaSuccess) e = M(5, cudaSuccess);
        return e;
    }
    if (e == cudaSuccess && small) {
        const bool front_quant = T <= moe::kFrontQuantMaxT;
        e = M(1, moe::launch_front(L, logits, ids, w, front_quant ? x : nullptr, T, s));
        if (e == cudaSuccess) e = M(2, front_quant ? cudaSuccess : moe::launch_quantize_scatter(L, x, T, s));
    } else {
        if (e == cudaSuccess && logits) e = moe::launch_route(L, logits, T, ids, w, s);
        if (e == cudaSuccess) e = M(1, moe::launch_permute(L, ids, T, L->offsets, L->row_src, L->row_dst, s));
        if (e == cudaSuccess) e = M(2, moe::launch_quantize_scatter(L, x, T, s));
    }
    cudaEvent_t mid = mark ? L->stage_ev[3] : nullptr;
    if (e == cudaSuccess) {
        if (tc) e = moe::launch_gemm_tc(L, T, s, mid, fuse_combine ? ids : nullptr, w, out);
        else e = moe::launch_gemm_cc(L, T, s, mid);
    }
    if (e == cudaSuccess) e = M(4, cudaSuccess);
    if (e == cudaSuccess) e = M(5, fuse_combine ? cudaSuccess : moe::launch_combine(L, ids, w, T, out, s));
    return e;
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_config* cfg) {
    if (check_config(cfg)) return 0;
    return workspace_bytes(*cfg);
}

const char* moe_last_error(const moe_layer* layer) {
    return layer ? layer->last_error : g_tls_error;
}

moe_status moe_create(const moe_config* cfg, const moe_weights* w, moe_stream_t stream,
                      moe_layer** out) {
    if (!out) return fail(nullptr, MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (const char* why = check_config(cfg)) return fail(nullptr, MOE_ERR_INVALID_ARG, "%s", why);
    if (!w) return fail(nullptr, MOE_ERR_INVALID_ARG, "weights is NULL");
    if (!w->gate_q || !w->gate_s || !w->up_q || !w->up_s || !w->down_q || !w->down_s)
        return fail(nullptr, MOE_ERR_INVALID_ARG, "a routed-expert weight pointer is NULL");
    if (cfg->weight_format == MOE_WEIGHTS_NVFP4 && (!w->gate_g || !w->up_g || !w->down_g))
        return fail(nullptr, MOE_ERR_INVALID_ARG, "NVFP4 weights need gate_g, up_g and down_g");
    if (cfg->has_shared && (!w->sh_gate_q || !w->sh_gate_s || !w->sh_up_q || !w->sh_up_s ||
                            !w->sh_down_q || !w->sh_down_s))
        return fail(nullptr, MOE_ERR_INVALID_ARG, "has_shared set but a shared weight pointer is NULL");

    moe_layer* L = new (std::nothrow) moe_layer;
    if (!L) return fail(nullptr, MOE_ERR_OOM, "host allocation failed");
    std::memset(L, 0, sizeof(*L));
    L->cfg = *cfg;
    L->cfg.has_shared = cfg->has_shared ? 1 : 0;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaGetDevice(&L->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device);
    if (e != cudaSuccess) {
        moe_status st = cuda_fail(nullptr, e, "device query");
        delete L;
        return st;
    }
    const moe_config& c = L->cfg;
    const size_t H = c.hidden, I = c.inter, E = c.n_experts, T = c.max_tokens, k = c.top_k;
    Sizes z = sizes_of(c);
    L->R_max = (int)z.R;
    L->Rp_max = (int)z.Rp;
    size_t total = 0;
    const bool nv = c.weight_format == MOE_WEIGHTS_NVFP4;
    const size_t sblk = nv ? 16 : 32;  // elements per weight block scale
    const size_t gq = E * I * H / 2, gs = E * I * H / sblk, dq = E * H * I / 2, ds = E * H * I / sblk;
    cudaError_t a = cudaSuccess;
    auto A = [&](auto** p, size_t bytes) { if (a == cudaSuccess) a = dalloc(p, bytes, &total); };
    A(&L->gu_q, 2 * gq); A(&L->gate_s, gs); A(&L->up_s, gs);
    A(&L->down_q, dq); A(&L->down_s, ds);
    A(&L->gu_sf, 2 * E * I * H / 32); A(&L->down_sf, E * H * I / 32);
    if (nv) { A(&L->gate_g, E * 4); A(&L->up_g, E * 4); A(&L->down_g, E * 4); }
    if (c.has_shared) {
        A(&L->sh_gu_q, 2 * I * H); A(&L->sh_gate_s, (I / 128) * (H / 128));
        A(&L->sh_up_s, (I / 128) * (H / 128));
        A(&L->sh_down_q, H * I); A(&L->sh_down_s, (H / 128) * (I / 128));
        A(&L->sh_gu_sf, 2 * I * H / 32); A(&L->sh_down_sf, H * I / 32);
    }
    A(&L->counts, E * 4); A(&L->offsets, (E + 1) * 4); A(&L->poff, (E + 1) * 4);
    A(&L->tile_scan, (E + 1) * 4); A(&L->chunk_scan, (E + 1) * 4);
    A(&L->row_src, z.R * 4); A(&L->row_dst, z.R * 4); A(&L->row_pos, z.R * 4);
    A(&L->pos_row, z.Rp * 4); A(&L->sh_desc, 8 * 4);
    A(&L->perm_cnt, (z.R + 1023) / 1024 * E * 4);
    A(&L->xq, z.Rp * H); A(&L->xs, z.Rp * H / 32);
    A(&L->hq, z.Rp * I); A(&L->hs, z.Rp * I / 32);
    A(&L->y, z.R * H * 4);
    if (c.has_shared) {
        A(&L->xq_tok, z.Tpad * H); A(&L->xs_tok, z.Tpad * H / 32);
        A(&L->hq_sh, z.Tpad * I); A(&L->hs_sh, z.Tpad * I / 32);
        A(&L->y_sh, T * H * 4);
    }
    A(&L->x_stage, T * H * 2); A(&L->logits_stage, T * E * 4); A(&L->out_stage, T * H * 4);
    A(&L->ids_stage, T * k * 4); A(&L->w_stage, T * k * 4);
    A(&L->d_err, 256);
    A(&L->sk_counters, (size_t)moe::kSkCounters(L) * 4);
    A(&L->sk_partials, (size_t)L->num_sms * 2 * 2 * 128 * 128 * 4);
    A(&L->dec_yw, (size_t)128 * 256 * 8);
    A(&L->gv_words, moe::gv_words_count(c, L->num_sms) * 4);
    if (a != cudaSuccess) {
        cudaGetLastError();
        free_all(L);
        delete L;
        return fail(nullptr, MOE_ERR_OOM, "device allocation of %zu bytes failed: %s", total,
                    cudaGetErrorString(a));
    }
    // weights: copy, then repack the block scales for the tensor-core kernels
    auto C = [&](void* dst, const void* src, size_t n) {
        if (a == cudaSuccess) a = cudaMemcpyAsync(dst, src, n, cudaMemcpyDefault, s);
    };
    // gate/up codes interleaved per 128 features (gate block, then up block)
    auto C2 = [&](void* dst, size_t dpitch, const void* src, size_t width, size_t height) {
        if (a == cudaSuccess)
            a = cudaMemcpy2DAsync(dst, dpitch, src, width, width, height, cudaMemcpyDefault, s);
    };
    const size_t blk = 128 * (H / 2);  // one 128-row block of fp4 codes
    C2(L->gu_q, 2 * blk, w->gate_q, blk, E * (I / 128));
    C2(L->gu_q + blk, 2 * blk, w->up_q, blk, E * (I / 128));
    C(L->gate_s, w->gate_s, gs); C(L->up_s, w->up_s, gs);
    C(L->down_q, w->down_q, dq); C(L->down_s, w->down_s, ds);
    if (nv) { C(L->gate_g, w->gate_g, E * 4); C(L->up_g, w->up_g, E * 4); C(L->down_g, w->down_g, E * 4); }
    if (c.has_shared) {
        C2(L->sh_gu_q, 2 * 128 * H, w->sh_gate_q, 128 * H, I / 128);
        C2(L->sh_gu_q + 128 * H, 2 * 128 * H, w->sh_up_q, 128 * H, I / 128);
        C(L->sh_gate_s, w->sh_gate_s, (I / 128) * (H / 128));
        C(L->sh_up_s, w->sh_up_s, (I / 128) * (H / 128));
        C(L->sh_down_q, w->sh_down_q, H * I); C(L->sh_down_s, w->sh_down_s, (H / 128) * (I / 128));
    }
    // (the tensor-core scale atoms exist for MXFP4 experts only)
    if (a == cudaSuccess && !nv)
        a = moe::pack_sf_pairs(L->gate_s, L->up_s, L->gu_sf, (int)E, (int)(I / 128), (int)H, 0, s);
    if (a == cudaSuccess && !nv)
        a = moe::pack_sf_pairs(L->down_s, nullptr, L->down_sf, (int)E, (int)(H / 256), (int)I, 1, s);
    if (c.has_shared) {
        if (a == cudaSuccess)
            a = moe::pack_sf_pairs(L->sh_gate_s, L->sh_up_s, L->sh_gu_sf, 1, (int)(I / 128), (int)H, 2, s);
        if (a == cudaSuccess)
            a = moe::pack_sf_pairs(L->sh_down_s, nullptr, L->sh_down_sf, 1, (int)(H / 256), (int)I, 3, s);
    }
    // a defined workspace: padding rows of the activation buffers read as zero
    // (and the epoch-tagged decode words start at epoch 0, which no launch uses)
    void* zero[] = {L->xq, L->xs, L->hq, L->hs, L->d_err, L->pos_row, L->sk_counters, L->dec_yw, L->gv_words};
    size_t zn[] = {z.Rp * H, z.Rp * H / 32, z.Rp * I, z.Rp * I / 32, 256, z.Rp * 4,
                   (size_t)moe::kSkCounters(L) * 4, (size_t)128 * 256 * 8, moe::gv_words_count(c, L->num_sms) * 4};
    for (int i = 0; i < 9 && a == cudaSuccess; ++i) a = cudaMemsetAsync(zero[i], 0, zn[i], s);
    if (c.has_shared) {
        void* zs[] = {L->xq_tok, L->xs_tok, L->hq_sh, L->hs_sh};
        size_t zsn[] = {z.Tpad * H, z.Tpad * H / 32, z.Tpad * I, z.Tpad * I / 32};
        for (int i = 0; i < 4 && a == cudaSuccess; ++i) a = cudaMemsetAsync(zs[i], 0, zsn[i], s);
    }
    if (a == cudaSuccess) a = cudaStreamSynchronize(s);
    if (a == cudaSuccess) a = moe::kernels_init();
    if (a == cudaSuccess) a = moe::cc_init();
    if (a == cudaSuccess) a = moe::tc_init(L);
    if (a == cudaSuccess) a = moe::gemv::init(L);
    if (a != cudaSuccess) {
        moe_status st = cuda_fail(nullptr, a, "moe_create");
        cudaGetLastError();
        free_all(L);
        delete L;
        return st;
    }
    L->gemm_path = 0;
    L->decode_kernel = 0;
    L->wait_ns = 2000000000ull;
    L->stall_next_decode = 0;
    L->prune_keep = L->cfg.top_k;
    L->prune_min_w = 0.f;
    L->prune_rho = 0.f;
    *out = L;
    return MOE_OK;
}

moe_status moe_destroy(moe_layer* layer) {
    if (!layer) return MOE_OK;
    free_all(layer);
    delete layer;
    return MOE_OK;
}

moe_status moe_set_stage_events(moe_layer* L, void* const* events, int n) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!events) { L->stage_ev_set = 0; return MOE_OK; }
    if (n != 6) return fail(L, MOE_ERR_INVALID_ARG, "n must be 6");
    for (int i = 0; i < 6; ++i) {
        if (!events[i]) return fail(L, MOE_ERR_INVALID_ARG, "event %d is NULL", i);
        L->stage_ev[i] = (cudaEvent_t)events[i];
    }
    L->stage_ev_set = 1;
    return MOE_OK;
}

unsigned long long moe_kernel_launches(const moe_layer* L) { return L ? L->launches : 0ull; }

moe_status moe_set_trace(moe_layer* L, unsigned long long* buf, size_t entries) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    // the GEMMs' and front kernel's counters, and the CUDA-core decode kernel's
    // per-CTA stamps followed by 4 x 256 event times
    const size_t ng = (size_t)48 * L->num_sms + 4, nd = (size_t)8 * L->num_sms + 1024;
    const size_t need = ng > nd ? ng : nd;
    if (buf && entries < need) return fail(L, MOE_ERR_INVALID_ARG, "trace buffer needs %zu entries", need);
    L->trace = buf;
    return MOE_OK;
}

moe_status moe_set_gemm_path(moe_layer* L, int path) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (path < 0 || path > 2) return fail(L, MOE_ERR_INVALID_ARG, "path must be 0, 1 or 2");
    if (path == 2 && !L->tc) return fail(L, MOE_ERR_UNSUPPORTED, "tensor-core path unavailable");
    L->gemm_path = path;
    return MOE_OK;
}

moe_status moe_set_route_prune(moe_layer* L, int keep, float min_w, float rho) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (keep < 1) return fail(L, MOE_ERR_INVALID_ARG, "keep must be >= 1");
    if (!std::isfinite(min_w)) return fail(L, MOE_ERR_INVALID_ARG, "min_w must be finite");
    if (!(rho >= 0.f && rho <= 1.f)) return fail(L, MOE_ERR_INVALID_ARG, "rho must be in [0, 1]");
    L->prune_keep = keep < L->cfg.top_k ? keep : L->cfg.top_k;
    L->prune_min_w = min_w;
    L->prune_rho = rho;
    return MOE_OK;
}

moe_status moe_set_wait_limit(moe_layer* L, double seconds) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!(seconds >= 1e-4 && seconds <= 60.0)) return fail(L, MOE_ERR_INVALID_ARG, "seconds must be in [1e-4, 60]");
    L->wait_ns = (uint64_t)(seconds * 1e9);
    return MOE_OK;
}

moe_status moe_test_stall_next_decode(moe_layer* L) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!moe::gemv::supported(L) && !(L->tc != nullptr && moe::decode_supported(L)))
        return fail(L, MOE_ERR_UNSUPPORTED, "the layer has no whole-layer decode kernel");
    L->stall_next_decode = 1;
    return MOE_OK;
}

moe_status moe_test_decode_split(int num_sms, int kept, int hidden, int inter, int nvfp4, int shared, int* cut) {
    if (num_sms < 1 || kept < 1 || hidden < 1024 || inter < 1024 || hidden % 1024 || inter % 1024 ||
        hidden > 8192 || inter > 8192 || !cut)
        return fail(nullptr, MOE_ERR_INVALID_ARG, "invalid split arguments");
    moe::gemv::split_table(num_sms, kept, hidden, inter, nvfp4 != 0, shared != 0, cut);
    return MOE_OK;
}

moe_status moe_set_decode_kernel(moe_layer* L, int kind) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (kind < 0 || kind > 2) return fail(L, MOE_ERR_INVALID_ARG, "kind must be 0, 1 or 2");
    if (kind == 1 && !moe::gemv::supported(L))
        return fail(L, MOE_ERR_UNSUPPORTED, "the layer's shape has no CUDA-core decode kernel");
    if (kind == 2 && !(L->tc != nullptr && moe::decode_supported(L)))
        return fail(L, MOE_ERR_UNSUPPORTED, "the layer's shape has no tcgen05 decode kernel");
    L->decode_kernel = kind;
    return MOE_OK;
}

moe_status moe_decode_info(const moe_layer* L, int* kind) {
    if (!L || !kind) return fail(nullptr, MOE_ERR_INVALID_ARG, "NULL pointer");
    *kind = decode_kind(L);
    return MOE_OK;
}

moe_status moe_route(moe_layer* L, const float* logits, int T, int32_t* ids, float* w,
                     moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!logits || !ids || !w) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (moe_status st = check_T(L, T)) return st;
    cudaError_t e = moe::launch_route(L, logits, T, ids, w, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_route");
}

moe_status moe_route_hash(moe_layer* L, const int32_t* token_ids, const int32_t* tid2eid, int V,
                          int T, int32_t* ids, float* w, moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!token_ids || !tid2eid || !ids || !w) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (V <= 0) return fail(L, MOE_ERR_INVALID_ARG, "V must be positive");
    if (moe_status st = check_T(L, T)) return st;
    cudaError_t e = moe::launch_route_hash(L, token_ids, tid2eid, V, T, ids, w, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_route_hash");
}

moe_status moe_permute(moe_layer* L, const int32_t* ids, int T, int32_t* offsets, int32_t* row_src,
                       int32_t* row_dst, moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!ids || !offsets || !row_src || !row_dst) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (moe_status st = check_T(L, T)) return st;
    cudaError_t e = moe::launch_permute(L, ids, T, offsets, row_src, row_dst, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_permute");
}

moe_status moe_quantize(moe_layer* L, const uint16_t* x, int T, uint8_t* q, uint8_t* s,
                        moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!x || !q || !s) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(x, 16) || !aligned(q, 8))
        return fail(L, MOE_ERR_INVALID_ARG, "x must be 16-byte and q 8-byte aligned");
    if (moe_status st = check_T(L, T)) return st;
    cudaError_t e = moe::launch_quantize_canonical(L, x, T, q, s, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_quantize");
}

moe_status moe_forward(moe_layer* L, const uint16_t* x, int T, const int32_t* ids, const float* w,
                       float* out, moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!x || !ids || !w || !out) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(x, 16) || !aligned(out, 16))
        return fail(L, MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    if (moe_status st = check_T(L, T)) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const bool ev = L->stage_ev_set != 0;
    L->stage_ev_set = 0;
    std::function<cudaError_t(int, cudaError_t)> mark = [&](int i, cudaError_t e) {
        return (ev && e == cudaSuccess) ? moe::record_stage(L->stage_ev[i], s) : e;
    };
    cudaError_t e = forward_kernels(L, nullptr, x, T, const_cast<int32_t*>(ids), const_cast<float*>(w),
                                    out, s, ev ? mark : std::function<cudaError_t(int, cudaError_t)>());
    L->trace = nullptr;
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_forward");
}

moe_status moe_route_forward(moe_layer* L, const float* logits, const uint16_t* x, int T, int32_t* ids,
                             float* w, float* out, moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!logits || !x || !ids || !w || !out) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(x, 16) || !aligned(out, 16))
        return fail(L, MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    if (moe_status st = check_T(L, T)) return st;
    const bool ev = L->stage_ev_set != 0;
    L->stage_ev_set = 0;
    cudaStream_t s = (cudaStream_t)stream;
    std::function<cudaError_t(int, cudaError_t)> mark = [&](int i, cudaError_t e) {
        return (ev && e == cudaSuccess) ? moe::record_stage(L->stage_ev[i], s) : e;
    };
    cudaError_t e = forward_kernels(L, logits, x, T, ids, w, out, s,
                                    ev ? mark : std::function<cudaError_t(int, cudaError_t)>());
    L->trace = nullptr;
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_route_forward");
}

moe_status moe_forward_host(moe_layer* L, const uint16_t* x, const float* logits, int T,
                            float* out, moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!x || !logits || !out) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (moe_status st = check_T(L, T)) return st;
    cudaStream_t s = (cudaStream_t)stream;
    // one token on the one-kernel decode path with page-locked buffers: the
    // kernel reads x and the logits and writes out in host memory directly
    // (mapped), so no copy is enqueued at all
    const int dk = T == 1 ? decode_kind(L) : 0;
    if (dk) {
        const void *dx = nullptr, *dl = nullptr, *dout = nullptr;
        if (mapped_host(x, &dx) && mapped_host(logits, &dl) && mapped_host(out, &dout) && aligned(dx, 16) &&
            aligned(dout, 16)) {
            L->stage_ev_set = 0;
            cudaError_t e = launch_decode_kind(L, dk, static_cast<const float*>(dl),
                                               static_cast<const uint16_t*>(dx), L->ids_stage, L->w_stage,
                                               static_cast<float*>(const_cast<void*>(dout)), s, true);
            L->trace = nullptr;
            return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_forward_host");
        }
    }
    const size_t H = L->cfg.hidden, E = L->cfg.n_experts;
    cudaError_t e = cudaMemcpyAsync(L->x_stage, x, (size_t)T * H * 2, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(L->logits_stage, logits, (size_t)T * E * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(L, e, "moe_forward_host: input copy");
    moe_status st = moe_route_forward(L, L->logits_stage, L->x_stage, T, L->ids_stage, L->w_stage,
                                      L->out_stage, stream);
    if (st != MOE_OK) return st;
    e = cudaMemcpyAsync(out, L->out_stage, (size_t)T * H * 4, cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_forward_host: output copy");
}

moe_status moe_hidden(moe_layer* L, int T, uint8_t* hq, uint8_t* hs, moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    if (!hq || !hs) return fail(L, MOE_ERR_INVALID_ARG, "NULL pointer");
    if (moe_status st = check_T(L, T)) return st;
    cudaError_t e = moe::launch_hidden_gather(L, T, hq, hs, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : cuda_fail(L, e, "moe_hidden");
}

moe_status moe_check(moe_layer* L, moe_stream_t stream) {
    if (!L) return fail(nullptr, MOE_ERR_INVALID_ARG, "layer is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    uint32_t flags = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&flags, L->d_err, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && flags) e = cudaMemset(L->d_err, 0, 4);
    if (e != cudaSuccess) return cuda_fail(L, e, "moe_check");
    if (flags & moe::ERR_TIMEOUT)
        return fail(L, MOE_ERR_TIMEOUT, "a device-side wait ran out of time (moe_set_wait_limit)");
    if (flags & moe::ERR_BAD_ID)
        return fail(L, MOE_ERR_INVALID_ARG, "an expert or token id was out of range");
    return MOE_OK;
}

}  // extern "C"
