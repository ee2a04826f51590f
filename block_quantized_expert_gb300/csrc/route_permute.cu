// route_permute.cu -- the integer and element-wise steps of the layer:
// learned and hash routing, the token -> expert counting sort, MXFP8
// quantisation of activations (scattered into the permuted row space), the
// fixed-order combine, and the one-time block-scale repack of the weights.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "layer.h"
#include "route.cuh"

namespace moe {

__global__ void __launch_bounds__(256) k_route(const float* __restrict__ logits, int T, int E,
                                               int k, float w_scale, RoutePrune prune,
                                               int32_t* __restrict__ ids, float* __restrict__ w,
                                               uint32_t* err) {
    pdl_launch_dependents();
    pdl_wait();
    const int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    route_token(logits + (size_t)t * E, E, k, w_scale, prune, ids + (size_t)t * k, w + (size_t)t * k, err,
                lane);
}

static RoutePrune route_prune_of(const moe_layer* L) {
    return RoutePrune{L->prune_keep, L->prune_min_w, L->prune_rho};
}

cudaError_t launch_route(moe_layer* L, const float* logits, int T, int32_t* ids, float* w,
                         cudaStream_t s) {
    const int warps_per_block = 8;
    dim3 grid((T + warps_per_block - 1) / warps_per_block);
    L->launches += 1;
    return launch_pdl(k_route, grid, dim3(32 * warps_per_block), 0, s, logits, T, L->cfg.n_experts,
                      L->cfg.top_k, L->cfg.w_scale, route_prune_of(L), ids, w, L->d_err);
}

// Hash-routed layers (guide, section 1: tid2eid maps a token id to its k
// experts; flat weights w_scale / k).
__global__ void k_route_hash(const int32_t* __restrict__ tok, const int32_t* __restrict__ tab,
                             int V, int T, int k, int E, float w_each, int32_t* __restrict__ ids,
                             float* __restrict__ w, uint32_t* err) {
    pdl_launch_dependents();
    pdl_wait();
    int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    int id = tok[t];
    bool ok = id >= 0 && id < V;
    for (int j = 0; j < k; ++j) {
        int e = ok ? tab[(size_t)id * k + j] : -1;
        if (e < 0 || e >= E) { e = -1; ok = false; }
        ids[(size_t)t * k + j] = e;
        w[(size_t)t * k + j] = w_each;
    }
    if (!ok) raise_flag(err, ERR_BAD_ID);
}

cudaError_t launch_route_hash(moe_layer* L, const int32_t* tok, const int32_t* tab, int V,
                              int T, int32_t* ids, float* w, cudaStream_t s) {
    float w_each = L->cfg.w_scale / (float)L->cfg.top_k;
    L->launches += 1;
    return launch_pdl(k_route_hash, dim3((T + 127) / 128), dim3(128), 0, s, tok, tab, V, T, L->cfg.top_k,
                      L->cfg.n_experts, w_each, ids, w, L->d_err);
}

// ---------------------------------------------------------------- permute --
// Block-wide exclusive scan of 4 ints per thread (1024 threads).
struct Int4Scan { int a, b, c, d; };

__device__ Int4Scan block_exclusive_scan4(Int4Scan v, Int4Scan* warp_tot, Int4Scan* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    Int4Scan inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int a = __shfl_up_sync(0xFFFFFFFFu, inc.a, o), b = __shfl_up_sync(0xFFFFFFFFu, inc.b, o);
        int c = __shfl_up_sync(0xFFFFFFFFu, inc.c, o), d = __shfl_up_sync(0xFFFFFFFFu, inc.d, o);
        if (lane >= o) { inc.a += a; inc.b += b; inc.c += c; inc.d += d; }
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        Int4Scan x = warp_tot[lane], xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int a = __shfl_up_sync(0xFFFFFFFFu, xi.a, o), b = __shfl_up_sync(0xFFFFFFFFu, xi.b, o);
            int c = __shfl_up_sync(0xFFFFFFFFu, xi.c, o), d = __shfl_up_sync(0xFFFFFFFFu, xi.d, o);
            if (lane >= o) { xi.a += a; xi.b += b; xi.c += c; xi.d += d; }
        }
        warp_tot[lane] = {xi.a - x.a, xi.b - x.b, xi.c - x.c, xi.d - x.d};
        if (lane == 31) *total = xi;
    }
    __syncthreads();
    Int4Scan base = warp_tot[warp];
    return {base.a + inc.a - v.a, base.b + inc.b - v.b, base.c + inc.c - v.c, base.d + inc.d - v.d};
}

// One chunk of the stable counting sort (1024 threads): rows [base, base +
// 1024) of R, each placed at its expert's start + cursor[e] (rows of e in
// earlier chunks) + rows of e in earlier warps of this chunk (per-warp counts
// wc) + in earlier lanes (match_any); cursor then advances by this chunk's
// counts.  Rows without a valid expert get row_dst = row_pos = -1.
__device__ void place_chunk(const int32_t* __restrict__ ids, int R, int E, int base, int* cursor,
                            const int* s_off, const int* s_poff, uint8_t* wc, int32_t* __restrict__ row_src,
                            int32_t* __restrict__ row_dst, int32_t* __restrict__ row_pos,
                            int32_t* __restrict__ pos_row) {
    // wc[e * 32 + w]: rows of expert e in warp w of this chunk (one byte each,
    // 32 contiguous bytes = 8 words per expert, summed four at a time)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* wcw = reinterpret_cast<uint32_t*>(wc);
    for (int i = tid; i < 8 * E; i += 1024) wcw[i] = 0u;
    __syncthreads();
    const int r = base + tid;
    int e = (r < R) ? ids[r] : -1;
    if (e >= E) e = -1;
    const unsigned grp = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(grp & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wc[e * 32 + warp] = (uint8_t)__popc(grp);
    __syncthreads();
    if (e >= 0) {
        // rows of e in warps 0 .. warp-1: whole words, then the low bytes of one
        int before = cursor[e] + rank;
        const uint32_t* we = wcw + e * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int lo = 4 * i;
            if (lo >= warp) break;
            uint32_t v = we[i];
            if (warp - lo < 4) v &= (1u << (8 * (warp - lo))) - 1u;
            before += (int)__dp4a(v, 0x01010101u, 0u);
        }
        const int p = s_off[e] + before, pp = s_poff[e] + before;
        row_src[p] = r;
        row_dst[r] = p;
        row_pos[r] = pp;
        pos_row[pp] = r;
    } else if (r < R) {
        row_dst[r] = -1;
        row_pos[r] = -1;
    }
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += 1024) {
        uint32_t add = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) add = __dp4a(wcw[e2 * 8 + i], 0x01010101u, add);
        cursor[e2] += (int)add;
    }
    __syncthreads();
}

// Stable counting sort of the rows r = t*k + j by expert, in one CTA of 1024
// threads: histogram, scan, then the rows in chunks of 1024 in ascending r,
// each row's rank = rows of the same expert in earlier chunks (cursor) +
// in earlier warps of this chunk (per-warp counts) + in earlier lanes
// (match_any).  Integer atomics only count, so the result is deterministic.
// Besides the ABI outputs it fills the padded bookkeeping of the GEMMs:
// every expert segment starts at a multiple of 128 rows.
__device__ void permute_body(
    const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_src, int32_t* __restrict__ row_dst, int32_t* __restrict__ counts,
    int32_t* __restrict__ poff, int32_t* __restrict__ tile_scan, int32_t* __restrict__ chunk_scan,
    int32_t* __restrict__ row_pos, int32_t* __restrict__ pos_row, int32_t* __restrict__ sh_desc,
    int T, uint32_t* err, int32_t* __restrict__ zero, int n_zero, int* dyn) {
    // dyn (shared): cnt, cursor, s_off, s_poff [E] each; then wc [32][E] bytes
    int* cnt = dyn;
    int* cursor = dyn + E;
    int* s_off = dyn + 2 * E;
    int* s_poff = dyn + 3 * E;
    uint8_t* wc = reinterpret_cast<uint8_t*>(dyn + 4 * E);
    __shared__ Int4Scan warp_tot[32];
    __shared__ Int4Scan total;
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < E; e += 1024) { cnt[e] = 0; cursor[e] = 0; }
    for (int i = tid; i < n_zero; i += 1024) zero[i] = 0;  // the GEMMs' split-tile counters
    if (tid == 0) bad = 0;
    __syncthreads();
    for (int r = tid; r < R; r += 1024) {
        int e = ids[r];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else if (e != -1) bad = 1;  // -1: an empty slot (pruned expert), left out quietly
    }
    __syncthreads();

    Int4Scan v = {0, 0, 0, 0};
    if (tid < E) {
        int n = cnt[tid];
        v = {n, (n + kRowTile - 1) / kRowTile * kRowTile, (n + kRowTile - 1) / kRowTile,
             (n + kChunk - 1) / kChunk};
    }
    Int4Scan ex = block_exclusive_scan4(v, warp_tot, &total);
    if (tid < E) {
        s_off[tid] = ex.a;
        s_poff[tid] = ex.b;
        offsets[tid] = ex.a;
        counts[tid] = v.a;
        poff[tid] = ex.b;
        tile_scan[tid] = ex.c;
        chunk_scan[tid] = ex.d;
    }
    if (tid == 0) {
        offsets[E] = total.a;
        poff[E] = total.b;
        tile_scan[E] = total.c;
        chunk_scan[E] = total.d;
        if (sh_desc) {  // the shared expert's single segment: all T tokens
            sh_desc[0] = T;
            sh_desc[1] = 0;
            sh_desc[2] = (T + kRowTile - 1) / kRowTile * kRowTile;
            sh_desc[3] = 0;
            sh_desc[4] = (T + kRowTile - 1) / kRowTile;
            sh_desc[5] = 0;
            sh_desc[6] = (T + kChunk - 1) / kChunk;
        }
        if (bad) raise_flag(err, ERR_BAD_ID);
    }
    __syncthreads();
    const int Rp = total.b;
    for (int p = tid; p < Rp; p += 1024) pos_row[p] = -1;

    for (int base = 0; base < R; base += 1024)
        place_chunk(ids, R, E, base, cursor, s_off, s_poff, wc, row_src, row_dst, row_pos, pos_row);
}

__global__ void __launch_bounds__(1024) k_permute(
    const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_src, int32_t* __restrict__ row_dst, int32_t* __restrict__ counts,
    int32_t* __restrict__ poff, int32_t* __restrict__ tile_scan, int32_t* __restrict__ chunk_scan,
    int32_t* __restrict__ row_pos, int32_t* __restrict__ pos_row, int32_t* __restrict__ sh_desc,
    int T, uint32_t* err, int32_t* __restrict__ zero, int n_zero) {
    extern __shared__ int dyn[];
    pdl_launch_dependents();
    pdl_wait();
    permute_body(ids, R, E, offsets, row_src, row_dst, counts, poff, tile_scan, chunk_scan, row_pos,
                 pos_row, sh_desc, T, err, zero, n_zero, dyn);
}

__global__ void k_perm_count(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ chunk_cnt);
__global__ void k_perm_place(const int32_t* __restrict__ ids, int R, int E, const int32_t* __restrict__ chunk_cnt,
                             int32_t* __restrict__ offsets, int32_t* __restrict__ row_src,
                             int32_t* __restrict__ row_dst, int32_t* __restrict__ counts,
                             int32_t* __restrict__ poff, int32_t* __restrict__ tile_scan,
                             int32_t* __restrict__ chunk_scan, int32_t* __restrict__ row_pos,
                             int32_t* __restrict__ pos_row, int32_t* __restrict__ sh_desc, int T, uint32_t* err,
                             int32_t* __restrict__ zero, int n_zero);

cudaError_t launch_permute(moe_layer* L, const int32_t* ids, int T, int32_t* offsets,
                           int32_t* row_src, int32_t* row_dst, cudaStream_t s) {
    const int R = T * L->cfg.top_k;
    const int E = L->cfg.n_experts;
    const size_t smem = (size_t)48 * E;
    if (R > 8 * 1024) {  // one CTA per 1024-row chunk (two launches: pays from about 8 chunks on)
        const int C = (R + 1023) / 1024;
        L->launches += 2;
        cudaError_t e = launch_pdl(k_perm_count, dim3(C), dim3(1024), (size_t)4 * E, s, ids, R, E,
                                   L->perm_cnt);
        if (e != cudaSuccess) return e;
        return launch_pdl(k_perm_place, dim3(C), dim3(1024), smem, s, ids, R, E,
                          (const int32_t*)L->perm_cnt, offsets, row_src, row_dst, L->counts, L->poff,
                          L->tile_scan, L->chunk_scan, L->row_pos, L->pos_row,
                          L->cfg.has_shared ? L->sh_desc : nullptr, T, L->d_err, L->sk_counters,
                          L->sk_counters ? kSkZeroed(L) : 0);
    }
    L->launches += 1;
    return launch_pdl(k_permute, dim3(1), dim3(1024), smem, s, ids, R, L->cfg.n_experts, offsets, row_src,
                      row_dst, L->counts, L->poff, L->tile_scan, L->chunk_scan, L->row_pos, L->pos_row,
                      L->cfg.has_shared ? L->sh_desc : nullptr, T, L->d_err, L->sk_counters,
                      L->sk_counters ? kSkZeroed(L) : 0);
}

// The same counting sort with caller-chosen bookkeeping buffers (no layer):
// counts [E], poff/tile_scan/chunk_scan [E+1], row_pos [T*k], pos_row [padded rows].
cudaError_t launch_permute_raw(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                               int32_t* row_src, int32_t* row_dst, int32_t* counts, int32_t* poff,
                               int32_t* tile_scan, int32_t* chunk_scan, int32_t* row_pos,
                               int32_t* pos_row, cudaStream_t s) {
    const size_t smem = (size_t)48 * E;
    k_permute<<<1, 1024, smem, s>>>(ids, T * k, E, offsets, row_src, row_dst, counts, poff, tile_scan,
                                 chunk_scan, row_pos, pos_row, nullptr, T, nullptr, nullptr, 0);
    return cudaGetLastError();
}



// The same sort over one CTA per 1024-row chunk (large batches), in two
// kernels: the chunks' expert counts, then every CTA scans them (its chunk's
// rows of expert e start after the rows of e in earlier chunks) and places
// its own rows with place_chunk.  The result is the one-CTA sort's.
__global__ void __launch_bounds__(1024) k_perm_count(const int32_t* __restrict__ ids, int R, int E,
                                                      int32_t* __restrict__ chunk_cnt) {
    extern __shared__ int sc[];  // [E]
    pdl_launch_dependents();
    pdl_wait();
    for (int e = threadIdx.x; e < E; e += 1024) sc[e] = 0;
    __syncthreads();
    const int r = blockIdx.x * 1024 + threadIdx.x;
    if (r < R) {
        const int e = ids[r];
        if (e >= 0 && e < E) atomicAdd(&sc[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += 1024) chunk_cnt[(size_t)blockIdx.x * E + e] = sc[e];
}

__global__ void __launch_bounds__(1024) k_perm_place(
    const int32_t* __restrict__ ids, int R, int E, const int32_t* __restrict__ chunk_cnt,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_src, int32_t* __restrict__ row_dst,
    int32_t* __restrict__ counts, int32_t* __restrict__ poff, int32_t* __restrict__ tile_scan,
    int32_t* __restrict__ chunk_scan, int32_t* __restrict__ row_pos, int32_t* __restrict__ pos_row,
    int32_t* __restrict__ sh_desc, int T, uint32_t* err, int32_t* __restrict__ zero, int n_zero) {
    extern __shared__ int dyn[];  // tot, cursor, s_off, s_poff [E]; wc [32][E] bytes
    int* tot = dyn;
    int* cursor = dyn + E;
    int* s_off = dyn + 2 * E;
    int* s_poff = dyn + 3 * E;
    uint8_t* wc = reinterpret_cast<uint8_t*>(dyn + 4 * E);
    __shared__ Int4Scan warp_tot[32];
    __shared__ Int4Scan total;
    __shared__ int bad;
    pdl_launch_dependents();
    pdl_wait();
    const int tid = threadIdx.x, C = gridDim.x, c = blockIdx.x;
    if (tid == 0) bad = 0;
    for (int e = tid; e < E; e += 1024) {
        int t = 0, b = 0;
        for (int cc = 0; cc < C; ++cc) {
            const int v = chunk_cnt[(size_t)cc * E + e];
            t += v;
            if (cc < c) b += v;
        }
        tot[e] = t;
        cursor[e] = b;
    }
    if (c == 0)
        for (int i = tid; i < n_zero; i += 1024) zero[i] = 0;  // the GEMMs' split-tile counters
    __syncthreads();
    {
        const int r = c * 1024 + tid;
        const int e = r < R ? ids[r] : -1;
        if (e != -1 && (e < 0 || e >= E)) bad = 1;  // -1: an empty slot, left out quietly
    }
    Int4Scan v = {0, 0, 0, 0};
    if (tid < E) {
        const int n = tot[tid];
        v = {n, (n + kRowTile - 1) / kRowTile * kRowTile, (n + kRowTile - 1) / kRowTile,
             (n + kChunk - 1) / kChunk};
    }
    Int4Scan ex = block_exclusive_scan4(v, warp_tot, &total);  // (its barriers order `bad` too)
    if (tid < E) {
        s_off[tid] = ex.a;
        s_poff[tid] = ex.b;
        if (c == 0) {
            offsets[tid] = ex.a;
            counts[tid] = v.a;
            poff[tid] = ex.b;
            tile_scan[tid] = ex.c;
            chunk_scan[tid] = ex.d;
        }
    }
    if (tid == 0) {
        if (c == 0) {
            offsets[E] = total.a;
            poff[E] = total.b;
            tile_scan[E] = total.c;
            chunk_scan[E] = total.d;
            if (sh_desc) {  // the shared expert's single segment: all T tokens
                sh_desc[0] = T;
                sh_desc[1] = 0;
                sh_desc[2] = (T + kRowTile - 1) / kRowTile * kRowTile;
                sh_desc[3] = 0;
                sh_desc[4] = (T + kRowTile - 1) / kRowTile;
                sh_desc[5] = 0;
                sh_desc[6] = (T + kChunk - 1) / kChunk;
            }
        }
        if (bad) raise_flag(err, ERR_BAD_ID);
    }
    __syncthreads();
    // the padding positions of every C-th expert segment read as no row
    for (int e = c; e < E; e += C) {
        const int lo = s_poff[e] + tot[e], hi = s_poff[e] + (tot[e] + kRowTile - 1) / kRowTile * kRowTile;
        for (int p = lo + tid; p < hi; p += 1024) pos_row[p] = -1;
    }
    place_chunk(ids, R, E, c * 1024, cursor, s_off, s_poff, wc, row_src, row_dst, row_pos, pos_row);
}

// --------------------------------------------------------------- quantise --
// MXFP8 of bf16 rows.  A group of 4 lanes owns one 32-block (8 elements per
// lane, one 16-byte load); the block amax is a 2-step shuffle max, the scale
// exponent comes from its fp32 exponent field, and the codes are the
// hardware's round-to-nearest-even, saturating e4m3 conversion of v * 2^-ex.
struct QuantDst {
    uint8_t* q;              // canonical [T][H] ...
    uint8_t* s;              // ... and [T][H/32]            (mode 0)
    uint8_t* xq;             // permuted rows [Rp][H] + atoms (mode 1)
    uint8_t* xs;
    const int32_t* row_pos;  // [T*k]
    int k;
    uint8_t* xq_tok;         // token-order rows [T][H] + atoms, or null
    uint8_t* xs_tok;
};

// One warp-task: 256 elements (8 blocks) of token row t; this lane's 8.
struct QTask {
    int t, b, h;
    bool active;
};

__device__ __forceinline__ QTask q_task(int H, int task, int lane) {
    const int tasks_per_row = (H + 255) / 256;
    QTask q;
    q.t = task / tasks_per_row;
    q.b = (task % tasks_per_row) * 8 + (lane >> 2);  // 32-block index
    q.active = q.b < H / 32;
    q.h = q.b * 32 + (lane & 3) * 8;
    return q;
}

__device__ __forceinline__ uint4 q_load(const uint16_t* __restrict__ x, int H, const QTask& q) {
    return q.active ? *reinterpret_cast<const uint4*>(x + (size_t)q.t * H + q.h) : make_uint4(0, 0, 0, 0);
}

// Quantise this lane's 8 elements (raw: their bf16 bits) and store them.
template <int kMode>
__device__ __forceinline__ void q_store(int H, const QuantDst& d, const QTask& q, uint4 raw, int lane) {
    const int t = q.t, b = q.b, h = q.h;
    const int part = lane & 3;
    const bool active = q.active;
    float v[8];
    float amax = 0.0f;
    if (active) {
        uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(wv[i] << 16);
            v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    if (!active) return;
    const int ex = mxfp8_exponent(amax);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        lo |= f32x2_to_e4m3x2(scale_pow2(v[2 * i], ex), scale_pow2(v[2 * i + 1], ex)) << (16 * i);
        hi |= f32x2_to_e4m3x2(scale_pow2(v[4 + 2 * i], ex), scale_pow2(v[5 + 2 * i], ex)) << (16 * i);
    }
    const uint2 codes = make_uint2(lo, hi);
    const uint8_t sbyte = (uint8_t)(ex + 127);
    if (kMode == 0) {
        *reinterpret_cast<uint2*>(d.q + (size_t)t * H + h) = codes;
        if (part == 0) d.s[(size_t)t * (H / 32) + b] = sbyte;
    } else {
        for (int j = 0; j < d.k; ++j) {
            const int p = d.row_pos[(size_t)t * d.k + j];
            if (p < 0) continue;
            *reinterpret_cast<uint2*>(d.xq + (size_t)p * H + h) = codes;
            if (part == 0) d.xs[sf_atom_offset(p, b, H)] = sbyte;
        }
        if (d.xq_tok) {
            *reinterpret_cast<uint2*>(d.xq_tok + (size_t)t * H + h) = codes;
            if (part == 0) d.xs_tok[sf_atom_offset(t, b, H)] = sbyte;
        }
    }
}

template <int kMode>
__device__ __forceinline__ void quantize_task(const uint16_t* __restrict__ x, int H, const QuantDst& d,
                                              int task, int lane) {
    const QTask q = q_task(H, task, lane);
    q_store<kMode>(H, d, q, q_load(x, H, q), lane);
}

template <int kMode>
__global__ void __launch_bounds__(256) k_quantize(const uint16_t* __restrict__ x, int T, int H,
                                                  QuantDst d) {
    pdl_launch_dependents();
    pdl_wait();
    const int task = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (task >= T * ((H + 255) / 256)) return;
    quantize_task<kMode>(x, H, d, task, threadIdx.x & 31);
}

// Small batches in one CTA (T <= kFrontMaxT): optional routing (one warp per
// token), the counting sort and (x non-null) the quantisation, each phase
// after a barrier.  Saves kernel boundaries on the decode path.
__global__ void __launch_bounds__(1024) k_front(
    const float* __restrict__ logits, float w_scale, RoutePrune prune, int32_t* __restrict__ ids,
    float* __restrict__ wts,
    const uint16_t* __restrict__ x, int T, int k, int E, int H, QuantDst qd, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_src, int32_t* __restrict__ row_dst, int32_t* __restrict__ counts,
    int32_t* __restrict__ poff, int32_t* __restrict__ tile_scan, int32_t* __restrict__ chunk_scan,
    int32_t* __restrict__ row_pos, int32_t* __restrict__ pos_row, int32_t* __restrict__ sh_desc,
    uint32_t* err, int32_t* __restrict__ zero, int n_zero, unsigned long long* trace) {
    extern __shared__ int dyn[];
    unsigned long long t_in = 0;
    if (trace && threadIdx.x == 0) t_in = tc_globaltimer();
    pdl_launch_dependents();
    pdl_wait();
    if (trace && threadIdx.x == 0) { trace[0] = t_in; trace[1] = tc_globaltimer(); }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (logits) {
        if (warp < T)
            route_token(logits + (size_t)warp * E, E, k, w_scale, prune, ids + (size_t)warp * k,
                        wts + (size_t)warp * k, err, lane);
        __syncthreads();
    }
    permute_body(ids, T * k, E, offsets, row_src, row_dst, counts, poff, tile_scan, chunk_scan, row_pos,
                 pos_row, sh_desc, T, err, zero, n_zero, dyn);
    __syncthreads();
    if (!x) {  // quantised by a grid-wide kernel after this one
        if (trace && threadIdx.x == 0) trace[2] = tc_globaltimer();
        return;
    }
    // the rows' padded positions, just written by this CTA, from shared
    // memory; each warp's x loads for up to kBatch tasks in flight at once
    __shared__ int32_t s_rp[kFrontMaxT * kMaxTopK];
    for (int r = threadIdx.x; r < T * k; r += blockDim.x) s_rp[r] = row_pos[r];
    __syncthreads();
    QuantDst qs = qd;
    qs.row_pos = s_rp;
    const int tasks = T * ((H + 255) / 256);
    constexpr int kBatch = 8;
    for (int base = warp; base < tasks; base += 32 * kBatch) {
        uint4 raw[kBatch];
        QTask qt[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int task = base + 32 * i;
            qt[i] = q_task(H, task < tasks ? task : 0, lane);
            qt[i].active = qt[i].active && task < tasks;
            raw[i] = q_load(x, H, qt[i]);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (base + 32 * i < tasks) q_store<1>(H, qs, qt[i], raw[i], lane);  // warp-uniform
    }
    if (trace) {
        __syncthreads();
        if (threadIdx.x == 0) trace[2] = tc_globaltimer();
    }
}

static cudaError_t quantize_launch(int mode, const uint16_t* x, int T, int H, QuantDst d,
                                   cudaStream_t s) {
    const long long tasks = (long long)T * ((H + 255) / 256);
    const int threads = 256;
    const long long blocks = (tasks * 32 + threads - 1) / threads;
    if (mode == 0) return launch_pdl(k_quantize<0>, dim3((unsigned)blocks), dim3(threads), 0, s, x, T, H, d);
    return launch_pdl(k_quantize<1>, dim3((unsigned)blocks), dim3(threads), 0, s, x, T, H, d);
}

cudaError_t launch_quantize_canonical(moe_layer* L, const uint16_t* x, int T, uint8_t* q,
                                      uint8_t* sc, cudaStream_t s) {
    L->launches += 1;
    QuantDst d{};
    d.q = q;
    d.s = sc;
    return quantize_launch(0, x, T, L->cfg.hidden, d, s);
}

cudaError_t launch_front(moe_layer* L, const float* logits, int32_t* ids, float* w, const uint16_t* x,
                         int T, cudaStream_t s) {
    QuantDst d{};
    d.xq = L->xq;
    d.xs = L->xs;
    d.row_pos = L->row_pos;
    d.k = L->cfg.top_k;
    if (L->cfg.has_shared) {
        d.xq_tok = L->xq_tok;
        d.xs_tok = L->xs_tok;
    }
    const size_t smem = (size_t)48 * L->cfg.n_experts;
    L->launches += 1;
    return launch_pdl(k_front, dim3(1), dim3(1024), smem, s, logits, L->cfg.w_scale, route_prune_of(L), ids, w,
                      x, T,
                      L->cfg.top_k, L->cfg.n_experts, L->cfg.hidden, d, L->offsets, L->row_src, L->row_dst,
                      L->counts, L->poff, L->tile_scan, L->chunk_scan, L->row_pos, L->pos_row,
                      L->cfg.has_shared ? L->sh_desc : nullptr, L->d_err, L->sk_counters,
                      L->sk_counters ? kSkZeroed(L) : 0,
                      L->trace ? L->trace + (size_t)4 * L->num_sms * 12 : nullptr);
}

cudaError_t launch_quantize_scatter(moe_layer* L, const uint16_t* x, int T, cudaStream_t s) {
    L->launches += 1;
    QuantDst d{};
    d.xq = L->xq;
    d.xs = L->xs;
    d.row_pos = L->row_pos;
    d.k = L->cfg.top_k;
    if (L->cfg.has_shared) {
        d.xq_tok = L->xq_tok;
        d.xs_tok = L->xs_tok;
    }
    return quantize_launch(1, x, T, L->cfg.hidden, d, s);
}

// ---------------------------------------------------------------- combine --
// out[t] = sum over the token's experts in ascending expert order (equal ids
// in j order) of w * y[row] (+ the shared expert): a fixed fp32 order, no
// atomics (guide, section 3.2, the FFN output equation).
// One thread per token and group of kCmbQ float4 columns, 128 features apart
// (every load of a warp is 512 contiguous bytes of one row; a warp covers
// 128 kCmbQ features, so H must be a multiple of that): the token's ids, row
// positions and weights are read once for them all.
template <int kCmbQ>
__global__ void __launch_bounds__(256) k_combine(const int32_t* __restrict__ ids,
                                                 const float* __restrict__ w,
                                                 const int32_t* __restrict__ row_pos,
                                                 const float* __restrict__ y,
                                                 const float* __restrict__ y_sh, int T, int H,
                                                 int k, float* __restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const int G = H / (4 * kCmbQ);  // column groups per token
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * G) return;
    const int t = (int)(i / G), g = (int)(i % G);
    const int c = (g / 32) * (128 * kCmbQ) + (g % 32) * 4;  // first column; then + 128 q
    int order[kMaxTopK];
    int idv[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        order[j] = j;
        idv[j] = (j < k) ? ids[(size_t)t * k + j] : INT_MAX;
    }
#pragma unroll
    for (int a = 1; a < kMaxTopK; ++a)
#pragma unroll
        for (int b = a; b > 0; --b)
            if (idv[order[b - 1]] > idv[order[b]]) {
                int tmp = order[b]; order[b] = order[b - 1]; order[b - 1] = tmp;
            }
    // every row's y and weight in flight at once (addresses in ascending
    // expert order), then summed in that order; a dropped row adds nothing
    bool live[kMaxTopK];
    float wv[kMaxTopK];
    int rr[kMaxTopK];
#pragma unroll
    for (int a = 0; a < kMaxTopK; ++a) {
        rr[a] = t * k + order[a];
        live[a] = a < k && row_pos[rr[a]] >= 0;
        wv[a] = live[a] ? w[rr[a]] : 0.f;
    }
    float4 acc[kCmbQ];
#pragma unroll
    for (int q = 0; q < kCmbQ; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int a = 0; a < kMaxTopK; ++a) {
        if (!live[a]) continue;
        float4 yv[kCmbQ];
#pragma unroll
        for (int q = 0; q < kCmbQ; ++q)
            yv[q] = *reinterpret_cast<const float4*>(y + (size_t)rr[a] * H + c + 128 * q);
        const float wt = wv[a];
#pragma unroll
        for (int q = 0; q < kCmbQ; ++q) {
            acc[q].x += wt * yv[q].x; acc[q].y += wt * yv[q].y; acc[q].z += wt * yv[q].z; acc[q].w += wt * yv[q].w;
        }
    }
    if (y_sh) {
#pragma unroll
        for (int q = 0; q < kCmbQ; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(y_sh + (size_t)t * H + c + 128 * q);
            acc[q].x += v.x; acc[q].y += v.y; acc[q].z += v.z; acc[q].w += v.w;
        }
    }
#pragma unroll
    for (int q = 0; q < kCmbQ; ++q) *reinterpret_cast<float4*>(out + (size_t)t * H + c + 128 * q) = acc[q];
}

cudaError_t launch_combine(moe_layer* L, const int32_t* ids, const float* w, int T,
                           float* out, cudaStream_t s) {
    const int H = L->cfg.hidden;  // a multiple of 256
    const int q = H % 512 == 0 ? 4 : 2;
    const long long n = (long long)T * (H / (4 * q));
    const dim3 grid((unsigned)((n + 255) / 256));
    L->launches += 1;
    const float* ysh = L->cfg.has_shared ? L->y_sh : nullptr;
    if (q == 4)
        return launch_pdl(k_combine<4>, grid, dim3(256), 0, s, ids, w, (const int32_t*)L->row_pos,
                          (const float*)L->y, ysh, T, H, L->cfg.top_k, out);
    return launch_pdl(k_combine<2>, grid, dim3(256), 0, s, ids, w, (const int32_t*)L->row_pos,
                      (const float*)L->y, ysh, T, H, L->cfg.top_k, out);
}

// ----------------------------------------------------------- test helpers --
__global__ void k_hidden_gather(const int32_t* __restrict__ row_pos, const uint8_t* __restrict__ hq,
                                const uint8_t* __restrict__ hs, int R, int I, uint8_t* __restrict__ oq,
                                uint8_t* __restrict__ os) {
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    if (r >= R) return;
    const int p = row_pos[r];
    for (int j = threadIdx.x; j < I; j += blockDim.x)
        oq[(size_t)r * I + j] = p >= 0 ? hq[(size_t)p * I + j] : 0;
    for (int b = threadIdx.x; b < I / 32; b += blockDim.x)
        os[(size_t)r * (I / 32) + b] = p >= 0 ? hs[sf_atom_offset(p, b, I)] : 0;
}

cudaError_t launch_hidden_gather(moe_layer* L, int T, uint8_t* hq, uint8_t* hs,
                                 cudaStream_t s) {
    const int R = T * L->cfg.top_k;
    k_hidden_gather<<<R, 256, 0, s>>>(L->row_pos, L->hq, L->hs, R, L->cfg.inter, hq, hs);
    L->launches += 1;
    return cudaGetLastError();
}

// Scale atoms of 256-row blocks: dst [mats][groups][K/128][2][512], byte
// (r % 32) * 16 + (r / 32) * 4 + kk of half h holds the scale of row r of that
// half and 32-block kt*4 + kk (one thread per byte).
__global__ void k_pack_sf_pairs(const uint8_t* __restrict__ srcA, const uint8_t* __restrict__ srcB,
                                uint8_t* __restrict__ dst, int groups, int K, int mode, long long n) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int KT = K / 128;
    const int o = (int)(i % 512), h = (int)((i / 512) % 2);
    const long long atom = i / 1024;  // (mat, group, kt)
    const int kt = (int)(atom % KT);
    const long long mg = atom / KT;
    const int g = (int)(mg % groups);
    const long long m = mg / groups;
    const int r = (o / 16) + 32 * ((o % 16) / 4), kk = o % 4;
    const int kb = kt * 4 + kk;
    uint8_t v;
    if (mode == 0) {
        const long long row = m * (long long)groups * 128 + (long long)g * 128 + r;
        v = (h ? srcB : srcA)[row * (K / 32) + kb];
    } else if (mode == 1) {
        const long long row = m * (long long)groups * 256 + (long long)(2 * g + h) * 128 + r;
        v = srcA[row * (K / 32) + kb];
    } else if (mode == 2) {
        v = (h ? srcB : srcA)[(long long)g * KT + kt];
    } else {
        v = srcA[(long long)(2 * g + h) * KT + kt];
    }
    dst[i] = v;
}

cudaError_t pack_sf_pairs(const uint8_t* srcA, const uint8_t* srcB, uint8_t* dst, int mats,
                          int groups, int K, int mode, cudaStream_t s) {
    const long long n = (long long)mats * groups * (K / 128) * 1024;
    k_pack_sf_pairs<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(srcA, srcB, dst, groups, K, mode, n);
    return cudaGetLastError();
}

// One shared-memory carveout for every kernel of the forward: the GEMMs need
// the maximum, and an SM whose carveout changes between two kernels must
// drain and reconfigure.
template <typename K>
static cudaError_t max_carveout(K kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

cudaError_t kernels_init() {
    cudaError_t e = cudaFuncSetAttribute(k_permute, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         48 * kMaxExperts);
    if (e == cudaSuccess) e = max_carveout(k_permute);
    if (e == cudaSuccess) e = max_carveout(k_route);
    if (e == cudaSuccess) e = max_carveout(k_route_hash);
    if (e == cudaSuccess) e = max_carveout(k_quantize<0>);
    if (e == cudaSuccess) e = max_carveout(k_quantize<1>);
    if (e == cudaSuccess) e = max_carveout(k_combine<2>);
    if (e == cudaSuccess) e = max_carveout(k_combine<4>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_perm_place, cudaFuncAttributeMaxDynamicSharedMemorySize, 48 * kMaxExperts);
    if (e == cudaSuccess) e = max_carveout(k_perm_place);
    if (e == cudaSuccess) e = max_carveout(k_perm_count);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_front, cudaFuncAttributeMaxDynamicSharedMemorySize, 48 * kMaxExperts);
    if (e == cudaSuccess) e = max_carveout(k_front);
    return e;
}

}  // namespace moe
