// gemm_tc.cu -- grouped expert GEMMs on the sm_103a block-scaled tensor cores
// (tcgen05.mma kind::mxf8f6f4, one UE8M0 scale per 32 K-elements).
//
// Orientation: weights are the MMA's A operand (M = 128 weight rows = output
// features), the routed tokens of one expert segment its B operand (N = 32..128
// token rows), so the fp32 accumulator D[feature][token] lives in tensor
// memory with one feature per TMEM lane.  MXFP4 weights are e2m1 (A format
// 5), the shared expert's fp8 weights e4m3 (A format 0); activations are
// e4m3.  Per 128-wide K step a TMA producer fills one pipeline stage with
// the weight tile(s) (fp4 unpacked by TMA into the 16-byte-aligned form the
// MMA reads), the token tile and three 512-byte scale-factor atoms; the MMA
// thread copies the atoms into tensor memory (tcgen05.cp) and issues four
// K=32 MMAs per accumulator; four epilogue warps read the accumulators back.
//
// Gate/up (guide, section 4): two accumulators (gate, up) per tile; the
// epilogue forms h = SiLU(g) * u in fp32 and requantises it to MXFP8 along
// the feature axis (32 features = one warp), writing h codes and scale atoms
// in the padded row space the down GEMM reads.  Down: one accumulator; the
// epilogue writes fp32 rows y[row][feature] for the fixed-order combine.
//
// Persistent grid of one CTA per SM; tiles enumerated (token tile u, weight
// tile m) with m fastest, so CTAs running together share a token tile and
// walk one expert's weights (L2 reuse).  Every wait is bounded in wall time:
// on expiry the CTA raises ERR_TIMEOUT, lets in-flight copies land, frees its
// tensor memory and exits.
#include <cuda.h>

#include <climits>
#include <new>

#include "common.cuh"
#include "layer.h"
#include "tc_ptx.cuh"

namespace moe {

using namespace tc;

// Transaction bytes of one 256-row weight copy: e2m1 codes unpacked by the
// TMA into 16-byte slots count the packed bytes (256 x 64), e4m3 256 x 128.
constexpr uint32_t kFp4BoxTx = 16384;
constexpr uint32_t kFp8BoxTx = 32768;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

struct TcArgs {
    int n_seg;
    const int32_t* counts;     // [n_seg] token rows per segment
    const int32_t* poff;       // [n_seg+1] padded row starts (multiples of 128)
    const int32_t* tile_scan;  // [n_seg+1] 128-row token tiles before segment e
    int K;                     // contraction length (multiple of 128)
    int N_out;                 // output features (multiple of 256 for down, 128 for gate/up)
    int mt;                    // 256-row weight blocks per segment
    int seg_rows;              // weight rows per segment (0: one shared matrix)
    const uint8_t* sfa;        // weight scale atom pairs [blocks][K/128][2][512]
    const uint8_t* sfb;        // activation scale atoms [Rp/128][K/128][512]
    uint8_t* hq;               // gate/up: h codes [Rp][N_out] + atoms
    uint8_t* hs;
    float* y;                  // down: y[row][N_out]
    const int32_t* pos_row;    // down: padded position -> y row (null: identity)
    uint32_t* err;
    uint32_t a_tx;             // TMA bytes of one 256-row weight copy
    int32_t* sk_cnt;           // [gridDim] arrival counters of cut tiles, by first CTA (start at 0)
    float* sk_part;            // [gridDim][2][2][128][128] partial accumulators
    unsigned long long* trace; // [gridDim][8] wait-time counters, or null
    // fused combine (down GEMM of small batches): after the last tile of a
    // 256-feature block, out[t][f] = sum over the token's experts in ascending
    // id order of w * y[t*k + j][f]
    const int32_t* cmb_ids;    // [T][k], or null (separate combine kernel)
    const float* cmb_w;        // [T][k]
    float* cmb_out;            // [T][N_out]
    const int32_t* cmb_row_pos;  // [T*k] padded position of row r (-1: dropped)
    int cmb_T, cmb_k;
    int32_t* cmb_cnt;          // [N_out / 256] tiles finished per block (start at 0)
};

// One pipeline stage: a 256-row weight tile (two 128-row MMA operands), up to
// 128 token rows, a pair of weight scale atoms and one activation scale atom.
struct TcCfg {
    static constexpr int kStages = 4;
    static constexpr int kABytes = 32768;  // 256 rows x 128 B (e2m1 in 16-byte slots, or e4m3)
    static constexpr int kBBytes = 16384;  // 128 rows x 128 B
    static constexpr int kSfOff = kABytes + kBBytes;
    static constexpr int kStageBytes = ((kSfOff + 1024 + 512) + 1023) / 1024 * 1024;
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kSmem = kBarOff + 256 + 1024;  // + barriers + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kAcc1Col = 128;
    static constexpr uint32_t kSfBase = 256;
    static constexpr uint32_t kSfPerStage = 12;  // A rows 0-127, A rows 128-255, B: 4 columns each
    static_assert(kSfBase + kStages * kSfPerStage <= kTmemCols, "tensor memory budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// warp 0: TMA, warp 1: MMA, warps 2-9: epilogue.  Ten warps put three on two
// of the four SM sub-partitions, whose 16K registers cap a thread at 168.
constexpr int kTcThreads = 320;
constexpr int kEpiWarps = 8;     // two per TMEM lane quarter, each half of the token columns

struct Tile {
    int e, n0, nvalid, nt, arow, f0, p0;
};

template <bool kGateUp>
__device__ __forceinline__ Tile decode_tile(const TcArgs& a, int t) {
    const int u = t / a.mt, m = t % a.mt;
    int lo = 0, hi = a.n_seg;  // segment with tile_scan[e] <= u < tile_scan[e+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.tile_scan + mid) <= u) lo = mid; else hi = mid;
    }
    Tile T;
    T.e = lo;
    T.n0 = (u - __ldg(a.tile_scan + lo)) * 128;
    T.nvalid = min(128, __ldg(a.counts + lo) - T.n0);
    T.nt = (T.nvalid + 31) & ~31;
    T.arow = a.seg_rows * lo + m * 256;
    T.f0 = m * (kGateUp ? 128 : 256);
    T.p0 = __ldg(a.poff + lo) + T.n0;
    return T;
}

// The work of one CTA: a sequence of (tile, K-stage range) segments.  With at
// least four waves of tiles, CTA c takes whole tiles c, c+G, ... (CTAs that
// run together share token tiles and one expert's weights in L2).  With
// fewer (decode), the tiles x K-stages space is cut into G equal contiguous
// ranges (stream-K), so every SM streams the same number of weight bytes; a
// tile cut between CTAs is finished by whichever of them arrives last,
// summing the partial accumulators in CTA (= K) order, so the result does
// not depend on arrival order.  A CTA range holds at most two cut pieces
// (its first and last segment), parked in slots 0 and 1.
struct Seg {
    int tile, kb0, kb1;
    int first_cta, last_cta;  // CTAs sharing this tile (equal: whole tile here)
};

struct SegIter {
    int tiles, KB, G, c;
    bool split;
    long long total, g, gend;
    int t;

    __device__ void init(int tiles_, int KB_, int G_, int c_) {
        tiles = tiles_; KB = KB_; G = G_; c = c_;
        total = (long long)tiles * KB;
        // fewer than four waves of whole tiles would leave SMs idle: split,
        // as long as every CTA still gets at least 4 K-stages
        split = tiles < 4 * G && total >= 4LL * G;
        if (split) { g = (long long)c * total / G; gend = (long long)(c + 1) * total / G; }
        t = c;
    }
    __device__ int owner(long long gs) const {  // CTA whose range holds global stage gs
        return (int)(((gs + 1) * G + total - 1) / total - 1);
    }
    __device__ long long range_begin(int cc) const { return (long long)cc * total / G; }
    __device__ bool next(Seg& s) {
        if (split) {
            if (g >= gend) return false;
            s.tile = (int)(g / KB);
            s.kb0 = (int)(g % KB);
            s.kb1 = (int)min((long long)KB, s.kb0 + (gend - g));
            s.first_cta = owner((long long)s.tile * KB);
            s.last_cta = owner((long long)s.tile * KB + KB - 1);
            g += s.kb1 - s.kb0;
            return true;
        }
        if (t >= tiles) return false;
        s.tile = t; s.kb0 = 0; s.kb1 = KB; s.first_cta = s.last_cta = c;
        t += G;
        return true;
    }
    // partial-accumulator slot of CTA cc's piece of `tile` (0: its first segment)
    __device__ int slot(int cc, int tile) const {
        return (int)(range_begin(cc) / KB) == tile ? 0 : 1;
    }
};

// Token n of a tile from its two accumulator values: gate/up -> h = SiLU(g) * u
// requantised to MXFP8 across the warp's 32 features; down -> two fp32 outputs.
template <bool kGateUp>
__device__ __forceinline__ void emit_token(const TcArgs& a, const Tile& T, int n, int q, int lane,
                                           float v0, float v1) {
    const int p = T.p0 + n;
    const int fm = 32 * q + lane;
    if (kGateUp) {
        const float h = silu_mul(v0, v1);
        const int ex = mxfp8_exponent(warp_max(fabsf(h)));
        const uint32_t code = f32x2_to_e4m3x2(scale_pow2(h, ex), 0.f) & 0xFFu;
        a.hq[(size_t)p * a.N_out + T.f0 + fm] = (uint8_t)code;
        if (lane == 0) a.hs[sf_atom_offset(p, (T.f0 + 32 * q) / 32, a.N_out)] = (uint8_t)(ex + 127);
    } else {
        const int row = a.pos_row ? __ldg(a.pos_row + p) : p;
        if (row >= 0) {
            float* yr = a.y + (size_t)row * a.N_out + T.f0;
            yr[fm] = v0;
            yr[128 + fm] = v1;
        }
    }
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Fused combine of features [f0, f0 + 256): epilogue thread i owns feature
// f0 + i; each token's experts are summed in ascending id order (equal ids in
// j order), the routing weight applied in fp32 -- the order of k_combine.
__device__ void combine_block(const TcArgs& a, int f0, int i) {
    const int k = a.cmb_k;
    for (int t = 0; t < a.cmb_T; ++t) {
        int order[kMaxTopK];
        int idv[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            order[j] = j;
            idv[j] = (j < k) ? __ldg(a.cmb_ids + (size_t)t * k + j) : INT_MAX;
        }
#pragma unroll
        for (int x = 1; x < kMaxTopK; ++x)
#pragma unroll
            for (int b = x; b > 0; --b)
                if (idv[order[b - 1]] > idv[order[b]]) {
                    const int tmp = order[b]; order[b] = order[b - 1]; order[b - 1] = tmp;
                }
        float acc = 0.f;
#pragma unroll
        for (int x = 0; x < kMaxTopK; ++x) {
            if (x < k) {
                const int r = t * k + order[x];
                if (__ldg(a.cmb_row_pos + r) < 0) continue;  // dropped row (bad id)
                acc += __ldg(a.cmb_w + r) * __ldcg(a.y + (size_t)r * a.N_out + f0 + i);
            }
        }
        a.cmb_out[(size_t)t * a.N_out + f0 + i] = acc;
    }
}

// Called by the 8 epilogue warps after they wrote the y rows of a finished
// tile of features [f0, f0 + 256): count the tile; the block's last tile
// combines the block.
__device__ __forceinline__ void tile_done_combine(const TcArgs& a, int f0, bool leader, volatile int* flag,
                                                  int warp, int lane) {
    __threadfence();
    epi_bar();
    if (leader) {
        const int ntiles = __ldg(a.tile_scan + a.n_seg);
        *flag = (atomicAdd(a.cmb_cnt + f0 / 256, 1) == ntiles - 1);
    }
    epi_bar();
    if (!*flag) return;
    __threadfence();
    combine_block(a, f0, (warp - 2) * 32 + lane);
}

// mbar_wait that adds the waited wall time to *acc when tracing.
__device__ __forceinline__ bool timed_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                           bool tr, unsigned long long& acc) {
    if (!tr) return mbar_wait(bar, parity, kWaitLimitNs, abort);
    const uint64_t t0 = globaltimer();
    const bool ok = mbar_wait(bar, parity, kWaitLimitNs, abort);
    acc += globaltimer() - t0;
    return ok;
}

template <bool kGateUp, uint32_t kAFmt>
__global__ void __launch_bounds__(kTcThreads, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB32,
          const __grid_constant__ CUtensorMap tmB64, const __grid_constant__ CUtensorMap tmB128,
          const TcArgs a) {
    using Cfg = TcCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (Cfg::kStages + s); };
    const uint32_t tmem_full = bar0 + 8u * (2 * Cfg::kStages);
    const uint32_t tmem_empty = tmem_full + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * Cfg::kStages + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = a.K / 128;
    const bool tr = a.trace != nullptr;
    unsigned long long* trc = tr ? a.trace + (size_t)blockIdx.x * 8 : nullptr;
    if (tr && threadIdx.x == 0) trc[0] = globaltimer();

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, kEpiWarps);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB32);
        prefetch_tmap(&tmB64);
        prefetch_tmap(&tmB128);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the prologue above overlaps the previous kernel; its outputs are read below
    pdl_launch_dependents();
    pdl_wait();
    const int tiles = __ldg(a.tile_scan + a.n_seg) * a.mt;

    auto give_up = [&]() {
        *abort_flag = 1;
        raise_flag(a.err, ERR_TIMEOUT);
    };
    SegIter it;
    it.init(tiles, KB, (int)gridDim.x, (int)blockIdx.x);
    Seg sg;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            unsigned long long w_empty = 0;
            while (ok && it.next(sg)) {
                const Tile T = decode_tile<kGateUp>(a, sg.tile);
                // one copy for the token rows: a 32-, 64- or 128-row box
                const CUtensorMap* tmB = T.nt == 32 ? &tmB32 : (T.nt == 64 ? &tmB64 : &tmB128);
                const uint32_t b_rows = T.nt == 32 ? 32u : (T.nt == 64 ? 64u : 128u);
                const uint32_t tx = a.a_tx + b_rows * 128u + 1024u + 512u;
                const size_t atom_a = (size_t)(T.arow / 256) * KB;
                const size_t atom_b = (size_t)(T.p0 / 128) * KB;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!timed_wait(empty_bar(stage), phase ^ 1u, abort_flag, tr, w_empty)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * Cfg::kStageBytes;
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, tx);
                    tma_load_2d(smem_u32(st), &tmA, kb * 128, T.arow, fb);
                    tma_load_2d(smem_u32(st + Cfg::kABytes), tmB, kb * 128, T.p0, fb);
                    bulk_load(smem_u32(st + Cfg::kSfOff), a.sfa + (atom_a + kb) * 1024, 1024, fb);
                    bulk_load(smem_u32(st + Cfg::kSfOff + 1024), a.sfb + (atom_b + kb) * 512, 512, fb);
                    if (++stage == Cfg::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (tr) trc[2] = w_empty;
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true;
            unsigned long long w_full = 0, w_acc = 0, n_stages = 0;
            while (ok && it.next(sg)) {
                const Tile T = decode_tile<kGateUp>(a, sg.tile);
                if (!timed_wait(tmem_empty, acc_phase ^ 1u, abort_flag, tr, w_acc)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!timed_wait(full_bar(stage), phase, abort_flag, tr, w_full)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    ++n_stages;
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + stage * Cfg::kStageBytes);
                    const uint32_t bt = st + Cfg::kABytes;
                    const uint32_t sf = st + Cfg::kSfOff;
                    const uint32_t sf_col = tmem + Cfg::kSfBase + stage * Cfg::kSfPerStage;
                    tmem_cp_32x128_x4(sf_col, desc_sf(sf));
                    tmem_cp_32x128_x4(sf_col + 4, desc_sf(sf + 512));
                    tmem_cp_32x128_x4(sf_col + 8, desc_sf(sf + 1024));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t id = idesc_mx(kAFmt, kFmtE4M3, 128, (uint32_t)T.nt, kk, kk);
                        const uint64_t bd = desc_sw128(bt + 32 * kk);
                        const uint32_t acc = (kb > sg.kb0 || kk) ? 1u : 0u;
                        mma_mx(tmem, desc_sw128(st + 32 * kk), bd, id, sf_col, sf_col + 8, acc);
                        mma_mx(tmem + Cfg::kAcc1Col, desc_sw128(st + 16384 + 32 * kk), bd, id, sf_col + 4,
                               sf_col + 8, acc);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == Cfg::kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tmem_full);
                acc_phase ^= 1u;
            }
            if (tr) { trc[3] = w_full; trc[4] = w_acc; trc[7] = n_stages; }
        }
    } else {
        // ---------------------------------------------------- epilogue --
        // Warp w (2..9) reads TMEM lanes of quarter w % 4 and token columns
        // [64 * h, 64 * h + 64), h = (w - 2) / 4: it copies both accumulators'
        // columns to registers, frees the accumulator for the next tile, and
        // only then does the SwiGLU / requantisation or the stores.
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int fm = 32 * q + lane;
        const int cb = 64 * hf;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)cb;
        const bool leader = warp == 2 && lane == 0;
        uint32_t acc_phase = 0;
        unsigned long long w_tf = 0, t_work = 0;
        while (it.next(sg)) {
            const Tile T = decode_tile<kGateUp>(a, sg.tile);
            if (!timed_wait(tmem_full, acc_phase, abort_flag, tr, w_tf)) {
                if (lane == 0) give_up();
                break;
            }
            const uint64_t tw0 = tr ? globaltimer() : 0;
            tc_fence_after();
            acc_phase ^= 1u;
            uint32_t v0[4][16], v1[4][16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (cb + 16 * j < T.nt) {  // warp-uniform
                    tmem_ld16(tq + 16 * j, v0[j]);
                    tmem_ld16(tq + Cfg::kAcc1Col + 16 * j, v1[j]);
                }
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty);
            const int nv = min(64, T.nvalid - cb);  // valid columns of this warp (may be <= 0)
            if (sg.first_cta == sg.last_cta) {
#pragma unroll
                for (int i = 0; i < 64; i += 4) {
                    if (i >= nv) break;  // warp-uniform
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (i + k < nv)
                            emit_token<kGateUp>(a, T, cb + i + k, q, lane, __uint_as_float(v0[(i + k) >> 4][(i + k) & 15]),
                                                __uint_as_float(v1[(i + k) >> 4][(i + k) & 15]));
                }
                if (!kGateUp && a.cmb_out) tile_done_combine(a, T.f0, leader, last_flag, warp, lane);
                if (tr) t_work += globaltimer() - tw0;
                continue;
            }
            // a piece of a split tile: park the partial sums, count arrivals
            float* part = a.sk_part + ((size_t)blockIdx.x * 2 + it.slot(blockIdx.x, sg.tile)) * 2 * 128 * 128;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                if (cb + i < T.nt) {
                    part[(size_t)(cb + i) * 128 + fm] = __uint_as_float(v0[i >> 4][i & 15]);
                    part[(size_t)(128 + cb + i) * 128 + fm] = __uint_as_float(v1[i >> 4][i & 15]);
                }
            }
            __threadfence();
            epi_bar();
            if (leader) {
                const int nparts = sg.last_cta - sg.first_cta + 1;
                *last_flag = (atomicAdd(a.sk_cnt + sg.first_cta, 1) == nparts - 1);
            }
            epi_bar();
            if (!*last_flag) continue;
            __threadfence();
            // the last piece to arrive sums all pieces in K order and finishes the tile
            for (int n = cb; n < min(T.nvalid, cb + 64); ++n) {
                float s0 = 0.f, s1 = 0.f;
                for (int cc = sg.first_cta; cc <= sg.last_cta; ++cc) {
                    const float* pp = a.sk_part + ((size_t)cc * 2 + it.slot(cc, sg.tile)) * 2 * 128 * 128;
                    s0 += __ldcg(pp + (size_t)n * 128 + fm);
                    s1 += __ldcg(pp + (size_t)(128 + n) * 128 + fm);
                }
                emit_token<kGateUp>(a, T, n, q, lane, s0, s1);
            }
            epi_bar();  // everyone has read the slots before the counter is reused
            if (leader) a.sk_cnt[sg.first_cta] = 0;
            if (!kGateUp && a.cmb_out) tile_done_combine(a, T.f0, leader, last_flag, warp, lane);
            if (tr) t_work += globaltimer() - tw0;
        }
        if (tr && leader) { trc[5] = w_tf; trc[6] = t_work; }
    }

    __syncthreads();
    if (tr && threadIdx.x == 0) trc[1] = globaltimer();
    if (*abort_flag) spin_ns(200000);  // copies / MMAs still in flight land first
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------------- host --
struct ActMaps {
    CUtensorMap b32, b64, b128;
};

struct TcState {
    CUtensorMap gu, down, sh_gu, sh_down;
    ActMaps xq, hq, xq_tok, hq_sh;
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D map over a row-major matrix [rows][cols] of 8-bit (fp4 = false) or
// packed 4-bit (fp4 = true) elements; box = 128 columns x box_rows rows,
// 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                     bool fp4) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {fp4 ? cols / 2 : cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool make_act_maps(ActMaps* m, const void* base, uint64_t cols, uint64_t rows) {
    return make_map(&m->b32, base, cols, rows, 32, false) && make_map(&m->b64, base, cols, rows, 64, false) &&
           make_map(&m->b128, base, cols, rows, 128, false);
}

template <bool G, uint32_t F>
static cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(k_gemm_tc<G, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::kSmem);
}

cudaError_t tc_init(moe_layer* L) {
    L->tc = nullptr;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, L->device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, L->device);
    if (major != 10 || minor != 3) return cudaSuccess;  // kernels are built for sm_103a only
    TcState* st = new (std::nothrow) TcState;
    if (!st) return cudaErrorMemoryAllocation;
    const uint64_t H = L->cfg.hidden, I = L->cfg.inter, E = L->cfg.n_experts;
    const uint64_t Rp = (uint64_t)L->Rp_max;
    const uint64_t Tpad = ((uint64_t)L->cfg.max_tokens + 127) / 128 * 128;
    bool ok = make_map(&st->gu, L->gu_q, H, E * 2 * I, 256, true) &&
              make_map(&st->down, L->down_q, I, E * H, 256, true) && make_act_maps(&st->xq, L->xq, H, Rp) &&
              make_act_maps(&st->hq, L->hq, I, Rp);
    if (ok && L->cfg.has_shared)
        ok = make_map(&st->sh_gu, L->sh_gu_q, H, 2 * I, 256, false) &&
             make_map(&st->sh_down, L->sh_down_q, I, H, 256, false) &&
             make_act_maps(&st->xq_tok, L->xq_tok, H, Tpad) && make_act_maps(&st->hq_sh, L->hq_sh, I, Tpad);
    if (!ok) {
        delete st;
        return cudaSuccess;  // no tensor-core path; the CUDA-core kernels run instead
    }
    cudaError_t e = set_smem_attr<true, kFmtE2M1>();
    if (e == cudaSuccess) e = set_smem_attr<false, kFmtE2M1>();
    if (e == cudaSuccess) e = set_smem_attr<true, kFmtE4M3>();
    if (e == cudaSuccess) e = set_smem_attr<false, kFmtE4M3>();
    if (e != cudaSuccess) {
        delete st;
        return e;
    }
    L->tc = st;
    return cudaSuccess;
}

void tc_free(moe_layer* L) {
    delete static_cast<TcState*>(L->tc);
    L->tc = nullptr;
}

template <bool G, uint32_t F>
static cudaError_t tc_launch(moe_layer* L, const CUtensorMap& a, const ActMaps& b, const TcArgs& args,
                             cudaStream_t s) {
    L->launches += 1;
    return launch_pdl(k_gemm_tc<G, F>, dim3(L->num_sms), dim3(kTcThreads), TcCfg::kSmem, s, a, b.b32, b.b64,
                      b.b128, args);
}

cudaError_t launch_gemm_tc(moe_layer* L, int T, cudaStream_t s, cudaEvent_t mid, const int32_t* cmb_ids,
                           const float* cmb_w, float* cmb_out) {
    const TcState* st = static_cast<const TcState*>(L->tc);
    const moe_config& c = L->cfg;
    TcArgs g{};
    g.n_seg = c.n_experts;
    g.counts = L->counts;
    g.poff = L->poff;
    g.tile_scan = L->tile_scan;
    g.K = c.hidden;
    g.N_out = c.inter;
    g.mt = c.inter / 128;
    g.seg_rows = 2 * c.inter;
    g.sfa = L->gu_sf;
    g.sfb = L->xs;
    g.hq = L->hq;
    g.hs = L->hs;
    g.err = L->d_err;
    g.a_tx = kFp4BoxTx;
    g.sk_part = L->sk_partials;
    g.sk_cnt = L->sk_counters;
    g.trace = L->trace;
    cudaError_t e = tc_launch<true, kFmtE2M1>(L, st->gu, st->xq, g, s);
    if (e == cudaSuccess && mid) e = cudaEventRecordWithFlags(mid, s, cudaEventRecordExternal);
    if (e != cudaSuccess) return e;
    TcArgs d = g;
    d.K = c.inter;
    d.N_out = c.hidden;
    d.mt = c.hidden / 256;
    d.seg_rows = c.hidden;
    d.sfa = L->down_sf;
    d.sfb = L->hs;
    d.hq = nullptr;
    d.hs = nullptr;
    d.y = L->y;
    d.pos_row = L->pos_row;
    d.sk_cnt = L->sk_counters + L->num_sms;
    if (cmb_ids) {
        d.cmb_ids = cmb_ids;
        d.cmb_w = cmb_w;
        d.cmb_out = cmb_out;
        d.cmb_row_pos = L->row_pos;
        d.cmb_T = T;
        d.cmb_k = c.top_k;
        d.cmb_cnt = L->sk_counters + 4 * L->num_sms;
    }
    d.trace = L->trace ? L->trace + (size_t)L->num_sms * 8 : nullptr;
    e = tc_launch<false, kFmtE2M1>(L, st->down, st->hq, d, s);
    if (e != cudaSuccess || !c.has_shared) return e;
    TcArgs sg = g;
    sg.n_seg = 1;
    sg.counts = L->sh_desc;
    sg.poff = L->sh_desc + 1;
    sg.tile_scan = L->sh_desc + 3;
    sg.seg_rows = 0;
    sg.sfa = L->sh_gu_sf;
    sg.sfb = L->xs_tok;
    sg.hq = L->hq_sh;
    sg.hs = L->hs_sh;
    sg.a_tx = kFp8BoxTx;
    sg.sk_cnt = L->sk_counters + 2 * L->num_sms;
    sg.trace = L->trace ? L->trace + (size_t)2 * L->num_sms * 8 : nullptr;
    e = tc_launch<true, kFmtE4M3>(L, st->sh_gu, st->xq_tok, sg, s);
    if (e != cudaSuccess) return e;
    TcArgs sd = sg;
    sd.K = c.inter;
    sd.N_out = c.hidden;
    sd.mt = c.hidden / 256;
    sd.sfa = L->sh_down_sf;
    sd.sfb = L->hs_sh;
    sd.hq = nullptr;
    sd.hs = nullptr;
    sd.y = L->y_sh;
    sd.pos_row = nullptr;
    sd.sk_cnt = L->sk_counters + 3 * L->num_sms;
    sd.trace = L->trace ? L->trace + (size_t)3 * L->num_sms * 8 : nullptr;
    return tc_launch<false, kFmtE4M3>(L, st->sh_down, st->hq_sh, sd, s);
}

}  // namespace moe
