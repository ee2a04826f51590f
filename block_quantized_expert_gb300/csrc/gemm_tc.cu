// gemm_tc.cu -- grouped expert GEMMs on the sm_103a block-scaled tensor cores
// (tcgen05.mma kind::mxf8f6f4, one UE8M0 scale per 32 K-elements).
//
// Orientation: the routed tokens of one expert segment are the MMA's A
// operand (M = 128 token rows) and a 256-row weight tile its B operand (N =
// 256), so one MMA per K=32 step covers the whole tile: the MMA cost is per
// instruction far more than per column (measured), and N = 256 is the
// widest shape.  The fp32 accumulator D[token][weight row] lives in tensor
// memory with one token row per TMEM lane.  Activations are e4m3; MXFP4
// weights are e2m1 (B format 5), the shared expert's fp8 weights e4m3 (B
// format 0).  Per 128-wide K step a TMA producer fills one pipeline stage
// with the weight tile (fp4 unpacked by TMA into the 16-byte-aligned form
// the MMA reads), the token rows (a 32-, 64- or 128-row box: rows past the
// box hold stale data whose accumulator rows are never read) and three
// 512-byte scale-factor atoms; the MMA thread copies the atoms into tensor
// memory (tcgen05.cp) and issues four K=32 MMAs; eight epilogue warps read
// the accumulator back, one token row per thread.
//
// Gate/up (guide, section 4): a weight tile is 128 gate rows and the
// matching 128 up rows, so a thread holds g and u of its token for 64
// features; it forms h = SiLU(g) * u in fp32 and requantises it to MXFP8
// along the feature axis (two 32-feature blocks, each within the thread),
// writing h codes and scale atoms in the padded row space the down GEMM
// reads.  Down: the epilogue writes fp32 rows y[row][feature] for the
// fixed-order combine.
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
#include "stage_event.h"
#include "route.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace tc;

// Transaction bytes of one 256-row weight copy: e2m1 codes unpacked by the
// TMA into 16-byte slots count the packed bytes (256 x 64), e4m3 256 x 128.
constexpr uint32_t kFp4BoxTx = 16384;
constexpr uint32_t kFp8BoxTx = 32768;

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
    uint64_t wait_ns;          // wall-time limit of every wait
    uint32_t a_tx;             // TMA bytes of one 256-row weight copy
    int32_t* sk_cnt;           // [gridDim] arrival counters of cut tiles, by first CTA (start at 0)
    float* sk_part;            // [gridDim][2][2][128][128] partial accumulators
    unsigned long long* trace; // [gridDim][12] timing counters, or null
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

// One pipeline stage: a 256-row weight tile (the B operand), up to 128 token
// rows (the A operand), a pair of weight scale atoms and one activation
// scale atom.
struct TcCfg {
    static constexpr int kStages = 4;
    static constexpr int kABytes = 32768;  // 256 rows x 128 B (e2m1 in 16-byte slots, or e4m3)
    static constexpr int kBBytes = 16384;  // 128 rows x 128 B
    static constexpr int kSfOff = kABytes + kBBytes;
    static constexpr int kStageBytes = ((kSfOff + 1024 + 512) + 1023) / 1024 * 1024;
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kSmem = kBarOff + 256 + 1024;  // + barriers + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kSfBase = 256;     // D: columns 0-255
    static constexpr uint32_t kSfPerStage = 12;  // tokens (A), weight rows 0-127, 128-255 (B): 4 columns each
    static_assert(kSfBase + kStages * kSfPerStage <= kTmemCols, "tensor memory budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// warp 0: TMA, warp 1: MMA, warps 2-9: epilogue.  Ten warps put three on two
// of the four SM sub-partitions, whose 16K registers cap a thread at 168.
constexpr int kTcThreads = 320;
constexpr int kEpiWarps = 8;     // two per TMEM lane quarter, each half of the weight columns

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
    // 32-bit arithmetic: a split happens only with fewer than 4 * G tiles of
    // at most 64 K-stages, so c * total stays below 2^23
    int tiles, KB, G, c;
    bool split;
    int total, g, gend;
    int t;

    __device__ void init(int tiles_, int KB_, int G_, int c_, int min_stages = 4) {
        tiles = tiles_; KB = KB_; G = G_; c = c_;
        total = tiles * KB;
        // fewer than four waves of whole tiles would leave SMs idle: split,
        // as long as every CTA still gets at least min_stages K-stages
        split = tiles < 4 * G && total >= min_stages * G;
        if (split) { g = c * total / G; gend = (c + 1) * total / G; }
        t = c;
    }
    __device__ int owner(int gs) const {  // CTA whose range holds global stage gs
        return ((gs + 1) * G + total - 1) / total - 1;
    }
    __device__ int range_begin(int cc) const { return cc * total / G; }
    __device__ bool next(Seg& s) {
        if (split) {
            if (g >= gend) return false;
            s.tile = g / KB;
            s.kb0 = g % KB;
            s.kb1 = min(KB, s.kb0 + (gend - g));
            s.first_cta = owner(s.tile * KB);
            s.last_cta = owner(s.tile * KB + KB - 1);
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
        return range_begin(cc) / KB == tile ? 0 : 1;
    }
};

// Token row n of a tile (one epilogue thread of column half hf) from its 128
// accumulator values.  Gate/up: v[0..63] are g and v[64..127] u of features
// f0 + 64 hf + (0..63); h = SiLU(g) * u is requantised to MXFP8 in two
// 32-feature blocks.  Down: v are the fp32 outputs f0 + 128 hf + (0..127).
template <bool kGateUp>
__device__ __forceinline__ void emit_row(const TcArgs& a, const Tile& T, int n, int hf, uint32_t (&v)[128]) {
    const int p = T.p0 + n;
    if (kGateUp) {
        const int fb = T.f0 + 64 * hf;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            // h replaces g in v[32 c .. 32 c + 31]
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float h = silu_mul(__uint_as_float(v[32 * c + j]), __uint_as_float(v[64 + 32 * c + j]));
                v[32 * c + j] = __float_as_uint(h);
                amax = fmaxf(amax, fabsf(h));
            }
            const int ex = mxfp8_exponent(amax);
            const uint32_t* h = v + 32 * c;
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[i] = f32x2_to_e4m3x2(scale_pow2(__uint_as_float(h[4 * i]), ex),
                                       scale_pow2(__uint_as_float(h[4 * i + 1]), ex)) |
                       (f32x2_to_e4m3x2(scale_pow2(__uint_as_float(h[4 * i + 2]), ex),
                                        scale_pow2(__uint_as_float(h[4 * i + 3]), ex)) << 16);
            st_global_v8(a.hq + (size_t)p * a.N_out + fb + 32 * c, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            a.hs[sf_atom_offset(p, (fb + 32 * c) / 32, a.N_out)] = (uint8_t)(ex + 127);
        }
    } else {
        const int row = a.pos_row ? __ldg(a.pos_row + p) : p;
        if (row >= 0) {
            // whole 32-byte sectors per store: each thread writes its own row
            float* yr = a.y + (size_t)row * a.N_out + T.f0 + 128 * hf;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                st_global_v8(yr + 8 * i, v[8 * i], v[8 * i + 1], v[8 * i + 2], v[8 * i + 3], v[8 * i + 4],
                             v[8 * i + 5], v[8 * i + 6], v[8 * i + 7]);
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
        float yv[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            order[j] = j;
            idv[j] = (j < k) ? __ldg(a.cmb_ids + (size_t)t * k + j) : INT_MAX;
            // every row's value in flight at once (a dropped row's y is not read)
            yv[j] = (j < k && __ldg(a.cmb_row_pos + t * k + j) >= 0)
                        ? __ldcg(a.y + (size_t)(t * k + j) * a.N_out + f0 + i)
                        : 0.f;
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
                if (__ldg(a.cmb_row_pos + r) < 0) continue;  // dropped row (bad id, empty slot)
                float v = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (j == order[x]) v = yv[j];
                acc += __ldg(a.cmb_w + r) * v;
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
    epi_bar();
    if (leader) a.cmb_cnt[f0 / 256] = 0;  // counters are left at zero
}

// mbar_wait (for at most limit_ns) that adds the waited wall time to *acc
// when tracing.
__device__ __forceinline__ bool timed_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                           bool tr, unsigned long long& acc, uint64_t limit_ns) {
    if (!tr) return mbar_wait(bar, parity, limit_ns, abort);
    const uint64_t t0 = globaltimer();
    const bool ok = mbar_wait(bar, parity, limit_ns, abort);
    acc += globaltimer() - t0;
    return ok;
}

// The producer and MMA roles run as whole warps (so every warp reaches the
// CTA-wide barriers converged): lane 0 waits and issues, the warp learns the
// outcome of each wait from it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, bool tr,
                                          unsigned long long& acc, int lane, uint64_t limit_ns) {
    int ok = 1;
    if (lane == 0) ok = timed_wait(bar, parity, abort, tr, acc, limit_ns) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
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
    unsigned long long* trc = tr ? a.trace + (size_t)blockIdx.x * 12 : nullptr;
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
    __syncwarp();  // warps reach CTA barriers converged (lane 0 may have run a role)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the prologue above overlaps the previous kernel; its outputs are read below
    pdl_launch_dependents();
    pdl_wait();
    if (tr && threadIdx.x == 0) trc[8] = globaltimer();
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
                if (!warp_wait(empty_bar(stage), phase ^ 1u, abort_flag, tr, w_empty, lane, a.wait_ns)) {
                    if (lane == 0) give_up();
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint8_t* st = smem + stage * Cfg::kStageBytes;
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, tx);
                    tma_load_2d(smem_u32(st), &tmA, kb * 128, T.arow, fb);
                    tma_load_2d(smem_u32(st + Cfg::kABytes), tmB, kb * 128, T.p0, fb);
                    bulk_load(smem_u32(st + Cfg::kSfOff), a.sfa + (atom_a + kb) * 1024, 1024, fb);
                    bulk_load(smem_u32(st + Cfg::kSfOff + 1024), a.sfb + (atom_b + kb) * 512, 512, fb);
                }
                if (++stage == Cfg::kStages) { stage = 0; phase ^= 1u; }
            }
        }
        if (tr && lane == 0) trc[2] = w_empty;
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        uint32_t stage = 0, phase = 0, acc_phase = 0;
        bool ok = true;
        unsigned long long w_full = 0, w_acc = 0, n_stages = 0;
        while (ok && it.next(sg)) {
            const Tile T = decode_tile<kGateUp>(a, sg.tile);
            if (!warp_wait(tmem_empty, acc_phase ^ 1u, abort_flag, tr, w_acc, lane, a.wait_ns)) {
                if (lane == 0) give_up();
                break;
            }
            for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                if (!warp_wait(full_bar(stage), phase, abort_flag, tr, w_full, lane, a.wait_ns)) {
                    if (lane == 0) give_up();
                    ok = false;
                    break;
                }
                ++n_stages;
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + stage * Cfg::kStageBytes);  // weights (B)
                    const uint32_t xt = st + Cfg::kABytes;                           // token rows (A)
                    const uint32_t sf = st + Cfg::kSfOff;
                    const uint32_t sf_col = tmem + Cfg::kSfBase + stage * Cfg::kSfPerStage;
                    tmem_cp_32x128_x4(sf_col, desc_sf(sf + 1024));     // token scales
                    tmem_cp_32x128_x4(sf_col + 4, desc_sf(sf));        // weight rows 0-127
                    tmem_cp_32x128_x4(sf_col + 8, desc_sf(sf + 512));  // weight rows 128-255
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t id = idesc_mx(kFmtE4M3, kAFmt, 128, 256, kk, kk);
                        const uint32_t acc = (kb > sg.kb0 || kk) ? 1u : 0u;
                        mma_mx(tmem, desc_sw128(xt + 32 * kk), desc_sw128(st + 32 * kk), id, sf_col, sf_col + 4, acc);
                    }
                    mma_commit(empty_bar(stage));
                }
                __syncwarp();
                if (++stage == Cfg::kStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) mma_commit(tmem_full);
            __syncwarp();
            acc_phase ^= 1u;
        }
        if (tr && lane == 0) { trc[3] = w_full; trc[4] = w_acc; trc[7] = n_stages; }
    } else {
        // ---------------------------------------------------- epilogue --
        // Warp w (2..9) reads TMEM lanes of quarter w % 4 (token rows n =
        // 32 (w % 4) + lane of the tile) and weight columns of half h = (w -
        // 2) / 4: gate/up -> gate columns 64 h .. + 63 and the matching up
        // columns 128 + 64 h .. + 63; down -> columns 128 h .. + 127.  It
        // copies them to registers, frees the accumulator for the next tile,
        // and only then does the SwiGLU / requantisation or the stores.
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int n = 32 * q + lane;
        const uint32_t c0 = kGateUp ? 64u * hf : 128u * hf;
        const uint32_t c1 = kGateUp ? 128u + 64u * hf : 128u * hf + 64u;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        const bool leader = warp == 2 && lane == 0;
        uint32_t acc_phase = 0;
        unsigned long long w_tf = 0, t_work = 0;
        while (it.next(sg)) {
            const Tile T = decode_tile<kGateUp>(a, sg.tile);
            // on a timeout the epilogue goes on with whatever the accumulator
            // holds (the error is raised), so all eight warps keep meeting at
            // the same named barriers
            if (!timed_wait(tmem_full, acc_phase, abort_flag, tr, w_tf, a.wait_ns) && lane == 0) give_up();
            const uint64_t tw0 = tr ? globaltimer() : 0;
            tc_fence_after();
            acc_phase ^= 1u;
            const bool rows_here = 32 * q < T.nvalid;  // warp-uniform: this quarter holds valid rows
            uint32_t v[128];  // fp32 bits
            if (rows_here) {
                tmem_ld32(tq + c0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(tq + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tmem_ld32(tq + c1, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
                tmem_ld32(tq + c1 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
                tmem_ld_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty);
            const bool valid = n < T.nvalid;
            if (sg.first_cta == sg.last_cta) {
                if (valid) emit_row<kGateUp>(a, T, n, hf, v);
                if (!kGateUp && a.cmb_out) tile_done_combine(a, T.f0, leader, last_flag, warp, lane);
                if (tr) t_work += globaltimer() - tw0;
                continue;
            }
            // a piece of a split tile: park the partial sums ([column][row]),
            // count arrivals
            float* part = a.sk_part + ((size_t)blockIdx.x * 2 + it.slot(blockIdx.x, sg.tile)) * 256 * 128;
            if (rows_here) {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    part[(size_t)(c0 + j) * 128 + n] = __uint_as_float(v[j]);
                    part[(size_t)(c1 + j) * 128 + n] = __uint_as_float(v[64 + j]);
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
            if (valid) {
                // the sums replace the parked values in v
#pragma unroll
                for (int j = 0; j < 128; ++j) v[j] = 0u;  // +0.0f
                for (int cc = sg.first_cta; cc <= sg.last_cta; ++cc) {
                    const float* pp = a.sk_part + ((size_t)cc * 2 + it.slot(cc, sg.tile)) * 256 * 128;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __ldcg(pp + (size_t)(c0 + j) * 128 + n));
                        v[64 + j] =
                            __float_as_uint(__uint_as_float(v[64 + j]) + __ldcg(pp + (size_t)(c1 + j) * 128 + n));
                    }
                }
                emit_row<kGateUp>(a, T, n, hf, v);
            }
            epi_bar();  // everyone has read the slots before the counter is reused
            if (leader) a.sk_cnt[sg.first_cta] = 0;
            if (!kGateUp && a.cmb_out) tile_done_combine(a, T.f0, leader, last_flag, warp, lane);
            if (tr) t_work += globaltimer() - tw0;
        }
        if (tr && leader) { trc[5] = w_tf; trc[6] = t_work; }
    }

    __syncwarp();  // the producer / MMA lane rejoins its warp before the CTA barrier
    __syncthreads();
    if (tr && threadIdx.x == 0) trc[1] = globaltimer();
    if (*abort_flag) spin_ns(200000);  // copies / MMAs still in flight land first
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// ------------------------------------------------------------- decode --
// The whole layer for one token (T = 1, learned router, no shared expert) in
// one cooperative kernel of one CTA per SM -- route, quantise, gate/up,
// down, combine -- so nothing of the token goes through a kernel boundary.
// Every CTA routes the token itself (ranks of the fp32 logits, the selection
// k_route makes, hence the same experts and weights everywhere) and
// quantises x straight into a resident shared-memory row.  The weights
// stream through a TMA / tcgen05 pipeline like k_gemm_tc's, split stream-K
// over all SMs.
//
// The k experts (ascending) may form groups whose phases run gate/up(0),
// gate/up(1), ..., down(0), down(1), ... so that one group's h hand-off
// overlaps the next group's streaming; with one accumulator the extra tile
// boundaries cost more than that saves (measured), so there is one group.
// The producer runs through all phases (the weights do not depend on h) and
// fetches the h of a group's experts once that group's first down weights are
// on their way.
//
// Cross-CTA hand-offs go through flags that hold the launch's epoch (a
// 64-bit launch counter that only grows), so nothing is ever reset: a tile
// cut between CTAs is finished by the CTA holding its first K-steps (it
// reaches that piece last), which adds the later pieces (parked by the
// following CTAs, which met them first) to its own; a gate/up tile's owner
// publishes h and an h flag; the owner of the last expert's tile of each
// 256-feature block waits for the other experts' y flags and writes the
// combined output.

// Orientation: with a single token the MMA cost is per instruction, not
// per column, so the weights are the B operand (N = 256: one MMA per K=32
// step covers a whole 256-row tile) and the token is the A operand (M =
// 128).  The token's codes are one contiguous row read through a no-swizzle
// K-major descriptor whose 16-byte K chunks are 16 bytes apart and whose
// 8-row groups all alias (stride 0): A rows 0, 8, ..., 120 are the token and
// the others are shifted copies, so TMEM lanes 0, 32, 64 and 96 each hold the
// token's outputs (one per lane quarter) and the other lanes are not read.
// D[lane][n] is weight row n of the tile: gate/up columns 0-127 are gate
// features, 128-255 the matching up features; down columns are 256 outputs.
constexpr int kDecStageBytes = 32768 + 1024;  // 256 weight rows + their scale atoms
constexpr int kDecStages = 6;
constexpr int kDecGroups = 1;
// stream-K split of a decode phase down to one K-stage per CTA: one kept
// expert has only 512 gate/up and 256 down stages for the whole grid
constexpr int kDecMinStages = 1;
constexpr int kDecSlotBytes = 2048 + 256;     // one h row (I <= 2048) + what the aliased rows reach
constexpr int kDecXOff = kDecStages * kDecStageBytes;            // the x row (H <= 4096) + reach
constexpr int kDecHOff = kDecXOff + 4096 + 512;                   // h rows [group][2 slots]
// Token scales: the source rows of the A scale copies, one 16-byte row per K
// step holding the step's four block scales once per lane quarter (the token
// rows 0, 32, 64, 96); a copy reads 512 bytes from its row.
constexpr int kDecXScaleBytes = 32 * 16 + 512;
constexpr int kDecHScaleBytes = 16 * 16 + 512;
constexpr int kDecTokScaleOff = kDecHOff + 2 * kDecGroups * kDecSlotBytes;  // x's, then h's [group][slot]
constexpr int kDecBarOff = kDecTokScaleOff + kDecXScaleBytes + 2 * kDecGroups * kDecHScaleBytes;
constexpr int kDecUpOff = kDecBarOff + 512;              // gate/up epilogue: the 128 up values of a tile
constexpr int kDecFrontOff = kDecUpOff + 512;            // routing: logits [E], candidates [<= 256] x 2
constexpr int kDecSmem = kDecFrontOff + 4096 + 2048 + 1024;
// tensor memory: D in columns 0-255; weight scales, 8 per stage; the
// token's scales of the down phases, 4 per stage; those of the gate/up
// phases, 4 per K step for every step (copied at the start, while the first
// weights are still in flight)
constexpr uint32_t kDecSfbCol = 256;
constexpr uint32_t kDecSfaStageCol = kDecSfbCol + 8 * kDecStages;
constexpr uint32_t kDecSfaResCol = kDecSfaStageCol + 4 * kDecStages;
static_assert(kDecSfaResCol + 4 * 32 <= 512, "tensor memory budget");
constexpr int kDecMaxTiles = 128;             // k * (I / 128) and k * (H / 256) for k <= 8, H <= 4096, I <= 2048
static_assert(kDecSmem <= 232448, "shared memory budget");
static_assert(kDecStageBytes % 1024 == 0, "128-byte swizzled weight tiles need 1024-byte alignment");

struct DecArgs {
    const float* logits;  // [E]
    const uint16_t* x;    // [H] bf16
    int E, k, H, I;       // k: the router's top-k (experts kept after pruning: DecCtx::k)
    float w_scale;
    RoutePrune prune;
    int32_t* ids_out;     // [k]
    float* w_out;         // [k]
    float* out;           // [H]
    const uint8_t* gu_sf;
    const uint8_t* down_sf;
    uint8_t* hq;          // [k][I] e4m3 (scratch)
    uint8_t* hs;          // [k][I/128][16] scale rows (scratch)
    unsigned long long* yw;  // [kDecMaxTiles][256] down tile outputs: epoch << 32 | fp32 bits
    float* sk_part;       // [G][2][2][128][128] partial accumulators of cut tiles
    unsigned long long* launches;  // launch counter: this launch's flags hold its value + 1
    uint32_t* piece_flag;  // [4 phases][G][2]: a cut tile's piece parked by CTA c in slot s
    uint32_t* h_flag;      // [kDecMaxTiles]: h of gate/up tile t written
    uint16_t* x_stage;     // x in host memory: CTA 0's device copy of it for the others, else null
    uint32_t* x_flag;      // x_stage written
    uint32_t* err;
    uint64_t wait_ns;      // wall-time limit of every wait
    // test hook: the h-flag waits expect a value no CTA writes (every CTA's
    // wait runs out after wait_ns; the call reports MOE_ERR_TIMEOUT)
    int stall_h;
    unsigned long long* trace;  // [gridDim][12] ns timestamps, or null
};

// One phase: the gate/up or down tiles of experts s_lo .. s_lo + n_s - 1
// (ascending order); idx = 2 * (down) + group names its flags and columns.
struct DecPhase {
    int s_lo, n_s, idx;
};

__device__ __forceinline__ int dec_groups(int k) { return k >= kDecGroups ? kDecGroups : 1; }

__device__ __forceinline__ DecPhase dec_phase(int k, bool down, int g) {
    const int G = dec_groups(k);
    const int lo = g * k / G, hi = (g + 1) * k / G;
    return DecPhase{lo, hi - lo, (down ? 2 : 0) + g};
}

// Shared state of one decode CTA.
struct DecCtx {
    uint8_t* smem;
    uint32_t bar0, tmem;
    uint32_t epoch;      // this launch's flag value
    int k;               // the experts kept (the router's top-k after tail pruning)
    volatile int* abort_flag;
    const int* seg_e;    // [k] experts, ascending
    const int* seg_j;    // [k] their position in the router output
    const float* seg_w;  // [k] their weights
    __device__ uint32_t full_bar(int st) const { return bar0 + 8u * st; }
    __device__ uint32_t empty_bar(int st) const { return bar0 + 8u * (kDecStages + st); }
    __device__ uint32_t tmem_full() const { return bar0 + 8u * (2 * kDecStages); }
    __device__ uint32_t tmem_empty() const { return bar0 + 8u * (2 * kDecStages) + 8u; }
    // a group's h rows and scale rows have landed
    __device__ uint32_t h_bar(int g) const { return bar0 + 8u * (2 * kDecStages) + 16u + 8u * g; }
    __device__ void give_up(const DecArgs& a) const {
        *abort_flag = 1;
        raise_flag(a.err, ERR_TIMEOUT);
    }
};

template <bool kGateUp>
__device__ __forceinline__ void dec_shape(const DecArgs& a, int& MT, int& KB, int& seg_rows) {
    MT = kGateUp ? a.I / 128 : a.H / 256;
    KB = (kGateUp ? a.H : a.I) / 128;
    seg_rows = kGateUp ? 2 * a.I : a.H;
}

// The (at most two) experts of this CTA's range of a down phase, in range
// order: slots[0], slots[1] (-1: none).  False if the range spans more.
__device__ bool dec_slots(const DecArgs& a, const DecPhase& ph, int (&slots)[2]) {
    int MT, KB, seg_rows;
    dec_shape<false>(a, MT, KB, seg_rows);
    SegIter it;
    it.init(ph.n_s * MT, KB, (int)gridDim.x, (int)blockIdx.x, kDecMinStages);
    Seg sg;
    int n = 0;
    slots[0] = slots[1] = -1;
    while (it.next(sg)) {  // ranges are contiguous: expert indices ascend
        const int sx = ph.s_lo + sg.tile / MT;
        if (n > 0 && slots[n - 1] == sx) continue;
        if (n == 2) return false;
        slots[n++] = sx;
    }
    return true;
}

// Warps 1-9 (all but the TMA producer).
__device__ __forceinline__ void work_bar() { asm volatile("bar.sync 2, 288;" ::: "memory"); }

// Publish / await a flag value.  A CTA publishes with a named barrier over
// its writers followed by one gpu-scope release store (cumulative over the
// writes the barrier ordered before it); a waiter's acquire load followed by
// a named barrier makes them visible to its whole CTA.  The wait gives up
// after limit_ns or when the CTA aborts.
__device__ __forceinline__ void flag_set(uint32_t* f, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t flag_get(const uint32_t* f) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
__device__ bool flag_wait(const uint32_t* f, uint32_t v, volatile int* abort, uint64_t limit_ns) {
    if (flag_get(f) == v) return true;
    const uint64_t t0 = globaltimer();
    while (flag_get(f) != v) {
        if (globaltimer() - t0 > limit_ns || *abort) return false;
        __nanosleep(32);
    }
    return true;
}

__device__ bool dec_fetch_h(const DecArgs& a, const DecCtx& c, const DecPhase& ph, int g, int lane);

// A value and its launch's epoch in one 64-bit word: a single-copy atomic
// store / load, so a reader that sees the epoch sees the value with it (no
// flag, no second round trip).
__device__ __forceinline__ void word_set(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long word_get(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// Wait (bounded by limit_ns, like flag_wait) until the n <= N words p[i * stride]
// carry epoch e, v[i] holding each word's first read.  Every round re-reads
// all words still of an earlier launch together: one round trip per round,
// not one per word.
template <int N>
__device__ bool words_wait(const unsigned long long* p, size_t stride, int n, uint32_t e, volatile int* abort,
                           uint64_t limit_ns, unsigned long long (&v)[N]) {
    const uint64_t t0 = globaltimer();
    while (true) {
        uint32_t pending = 0;
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (i < n && (uint32_t)(v[i] >> 32) != e) pending |= 1u << i;
        if (!pending) return true;
        if (globaltimer() - t0 > limit_ns || *abort) return false;
        __nanosleep(32);
#pragma unroll
        for (int i = 0; i < N; ++i)
            if ((pending >> i) & 1u) v[i] = word_get(p + (size_t)i * stride);
    }
}

// TMA producer (warp 0; lane 0 waits and issues): the weight tiles and
// scale atoms of this CTA's stream-K range of one phase, into the ring.  A
// down phase fetches group g's h after its first kDecStages weight loads:
// those land during the gate/up -> down hand-off (the weights do not depend
// on h), so the down MMAs find a full ring when h arrives.
template <bool kGateUp>
__device__ bool dec_produce(const DecArgs& a, const DecCtx& c, const CUtensorMap* tmA, const DecPhase& ph, int g,
                            uint32_t& stage, uint32_t& phase, int lane) {
    int MT, KB, seg_rows;
    dec_shape<kGateUp>(a, MT, KB, seg_rows);
    const uint8_t* sfa = kGateUp ? a.gu_sf : a.down_sf;
    SegIter it;
    it.init(ph.n_s * MT, KB, (int)gridDim.x, (int)blockIdx.x, kDecMinStages);
    Seg sg;
    int issued = 0;
    bool h_done = kGateUp;
    while (it.next(sg)) {
        const int s = ph.s_lo + sg.tile / MT, m = sg.tile % MT;
        const int arow = c.seg_e[s] * seg_rows + m * 256;
        const size_t atom_a = (size_t)(arow / 256) * KB;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
            if (!h_done && issued == kDecStages) {
                if (!dec_fetch_h(a, c, ph, g, lane)) return false;
                h_done = true;
            }
            ++issued;
            unsigned long long none = 0;
            if (!warp_wait(c.empty_bar(stage), phase ^ 1u, c.abort_flag, false, none, lane, a.wait_ns)) {
                if (lane == 0) c.give_up(a);
                return false;
            }
            if (lane == 0) {
                uint8_t* st = c.smem + stage * kDecStageBytes;
                const uint32_t fb = c.full_bar(stage);
                mbar_arrive_expect_tx(fb, kFp4BoxTx + 1024u);
                tma_load_2d(smem_u32(st), tmA, kb * 128, arow, fb);
                bulk_load(smem_u32(st + 32768), sfa + (atom_a + kb) * 1024, 1024, fb);
            }
            if (++stage == kDecStages) { stage = 0; phase ^= 1u; }
        }
    }
    return h_done || dec_fetch_h(a, c, ph, g, lane);
}

// Before a down phase's MMAs (producer warp): wait for the h flags of the
// phase's experts in this CTA's range (their gate/up tiles, I / 128 <= 16
// each), then bring their h rows and scale rows in with bulk copies that
// complete on the group's h barrier.
__device__ bool dec_fetch_h(const DecArgs& a, const DecCtx& c, const DecPhase& ph, int g, int lane) {
    int slots[2];
    if (!dec_slots(a, ph, slots)) {  // more than two experts in one range: not supported
        if (lane == 0) c.give_up(a);
        return false;
    }
    const int mt_gu = a.I / 128;  // lanes 0-15 slot 0, 16-31 slot 1
    const int sx = slots[lane >> 4];
    bool ok = true;
    // (stall_h: a value no launch writes -- the test of the bounded waits)
    const uint32_t want = a.stall_h ? (c.epoch ^ 0x80000000u) : c.epoch;
    if (sx >= 0 && (lane & 15) < mt_gu) ok = flag_wait(a.h_flag + sx * mt_gu + (lane & 15), want, c.abort_flag, a.wait_ns);
    if (!__all_sync(0xFFFFFFFFu, ok)) {
        if (lane == 0) c.give_up(a);
        return false;
    }
    if (lane == 0) {
        // the copies read global memory other CTAs wrote through the generic proxy
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const uint32_t hb = c.h_bar(g);
        const uint32_t srow = (uint32_t)mt_gu * 16;
        const int nsl = slots[1] >= 0 ? 2 : 1;
        mbar_arrive_expect_tx(hb, (uint32_t)nsl * ((uint32_t)a.I + srow));
        for (int sl = 0; sl < nsl; ++sl) {
            bulk_load(smem_u32(c.smem + kDecHOff + (2 * g + sl) * kDecSlotBytes), a.hq + (size_t)slots[sl] * a.I,
                      (uint32_t)a.I, hb);
            bulk_load(smem_u32(c.smem + kDecTokScaleOff + kDecXScaleBytes + (2 * g + sl) * kDecHScaleBytes),
                      a.hs + (size_t)slots[sl] * srow, srow, hb);
        }
    }
    __syncwarp();
    return true;
}

// MMA issuer (warp 1; lane 0 waits and issues): per K=32 step one M = 128,
// N = 256 MMA of the resident token row against the streamed weight tile.
template <bool kGateUp>
__device__ bool dec_mma(const DecArgs& a, const DecCtx& c, const DecPhase& ph, int g, uint32_t& stage,
                        uint32_t& phase, uint32_t& acc_phase, int lane) {
    int MT, KB, seg_rows;
    dec_shape<kGateUp>(a, MT, KB, seg_rows);
    const uint32_t tok_base = smem_u32(c.smem + kDecTokScaleOff);
    unsigned long long none = 0;
    int slots[2] = {-1, -1};
    if (kGateUp) {
        if (g == 0) {  // x's scales for every K step, once
            if (lane == 0) {
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb)
                    tmem_cp_32x128_x4(c.tmem + kDecSfaResCol + kb * 4, desc_sf(tok_base + kb * 16));
            }
            __syncwarp();
        }
    } else {
        dec_slots(a, ph, slots);
        if (!warp_wait(c.h_bar(g), 0, c.abort_flag, false, none, lane, a.wait_ns)) {  // the group's h rows
            if (lane == 0) c.give_up(a);
            return false;
        }
    }
    SegIter it;
    it.init(ph.n_s * MT, KB, (int)gridDim.x, (int)blockIdx.x, kDecMinStages);
    Seg sg;
    while (it.next(sg)) {
        const int s = ph.s_lo + sg.tile / MT;
        const int sl = (!kGateUp && slots[1] == s) ? 1 : 0;
        const uint32_t a_base = kGateUp ? smem_u32(c.smem + kDecXOff)
                                        : smem_u32(c.smem + kDecHOff + (2 * g + sl) * kDecSlotBytes);
        const uint32_t sa_base = tok_base + kDecXScaleBytes + (2 * g + sl) * kDecHScaleBytes;
        if (!warp_wait(c.tmem_empty(), acc_phase ^ 1u, c.abort_flag, false, none, lane, a.wait_ns)) {
            if (lane == 0) c.give_up(a);
            return false;
        }
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
            if (!warp_wait(c.full_bar(stage), phase, c.abort_flag, false, none, lane, a.wait_ns)) {
                if (lane == 0) c.give_up(a);
                return false;
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t st = smem_u32(c.smem + stage * kDecStageBytes);
                const uint32_t sfb_col = c.tmem + kDecSfbCol + stage * 8;  // weight rows 0-127, 128-255
                const uint32_t at = a_base + kb * 128;
                uint32_t sfa_col = c.tmem + kDecSfaResCol + kb * 4;
                if (!kGateUp) {
                    sfa_col = c.tmem + kDecSfaStageCol + stage * 4;
                    tmem_cp_32x128_x4(sfa_col, desc_sf(sa_base + kb * 16));
                }
                tmem_cp_32x128_x4(sfb_col, desc_sf(st + 32768));
                tmem_cp_32x128_x4(sfb_col + 4, desc_sf(st + 32768 + 512));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t id = idesc_mx(kFmtE4M3, kFmtE2M1, 128, 256, kk, kk);
                    const uint32_t acc = (kb > sg.kb0 || kk) ? 1u : 0u;
                    mma_mx(c.tmem, smem_desc(at + 32 * kk, 16, 0, 0), desc_sw128(st + 32 * kk), id, sfa_col,
                           sfb_col, acc);
                }
                mma_commit(c.empty_bar(stage));
            }
            __syncwarp();
            if (++stage == kDecStages) { stage = 0; phase ^= 1u; }
        }
        if (lane == 0) mma_commit(c.tmem_full());
        __syncwarp();
        acc_phase ^= 1u;
    }
    return true;
}

// Epilogue (warps 2-9): warp w takes D columns 32 (w - 2) .. + 31 from the
// token lane of its lane quarter (lane 0 of the warp reads them, the warp
// shares them out: thread t gets column 32 (w - 2) + t).  Gate/up: warps 6-9
// hand their up values to warps 2-5 through shared memory, which form h =
// SiLU(g) * u and requantise it to MXFP8 (32 features = one warp).  Down: y,
// or for the last expert's tile of a feature block the combined output.
template <bool kGateUp>
__device__ void dec_epilogue(const DecArgs& a, const DecCtx& c, const DecPhase& ph, uint32_t& acc_phase) {
    int MT, KB, seg_rows;
    dec_shape<kGateUp>(a, MT, KB, seg_rows);
    uint32_t* pflag = a.piece_flag + ph.idx * 2 * gridDim.x;
    const int pcol = ph.idx * 256;  // the phases park pieces in different columns
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int col = 32 * (warp - 2) + lane;  // this thread's D column (0-255)
    const uint32_t taddr = c.tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * (warp - 2));
    float* up_s = reinterpret_cast<float*>(c.smem + kDecUpOff);
    const bool lead_warp = warp == 2;
    SegIter it;
    it.init(ph.n_s * MT, KB, (int)gridDim.x, (int)blockIdx.x, kDecMinStages);
    Seg sg;
    while (it.next(sg)) {
        const int s = ph.s_lo + sg.tile / MT, m = sg.tile % MT;
        const int gt = s * MT + m;  // the tile's index over all experts (its flags)
        const int f0 = m * (kGateUp ? 128 : 256);
        const bool split = sg.first_cta != sg.last_cta;
        const bool owner = !split || (int)blockIdx.x == sg.first_cta;
        float later = 0.f;  // the later pieces of a cut tile this CTA finishes, in K order
        if (split && owner) {
            // they come from the following CTAs, which met them first: wait
            // for them and load them while this CTA's own MMAs still run (the
            // piece is this CTA's last of the phase, so no later tile waits
            // for the accumulator meanwhile)
            if (lead_warp) {
                bool ok = true;
                const int cc = sg.first_cta + 1 + lane;
                if (cc <= sg.last_cta) ok = flag_wait(pflag + cc * 2 + it.slot(cc, sg.tile), c.epoch, c.abort_flag, a.wait_ns);
                if (!__all_sync(0xFFFFFFFFu, ok) && lane == 0) c.give_up(a);
            }
            epi_bar();  // the acquire loads above make the pieces visible to the CTA
            for (int cc = sg.first_cta + 1; cc <= sg.last_cta; ++cc)
                later += __ldcg(a.sk_part + ((size_t)cc * 2 + it.slot(cc, sg.tile)) * 2 * 128 * 128 + pcol + col);
        }
        // on a timeout the epilogue goes on with whatever the accumulator
        // holds (the error is raised), so all eight warps keep meeting at
        // the same named barriers
        if (!mbar_wait(c.tmem_full(), acc_phase, a.wait_ns, c.abort_flag) && lane == 0) c.give_up(a);
        tc_fence_after();
        acc_phase ^= 1u;
        uint32_t r[32];
        tmem_ld32(taddr, r);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(c.tmem_empty());
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float x = __shfl_sync(0xFFFFFFFFu, __uint_as_float(r[i]), 0);
            if (lane == i) v = x;
        }
        if (!owner) {
            // a later piece: park it and go on
            const int slot = it.slot(blockIdx.x, sg.tile);
            a.sk_part[((size_t)blockIdx.x * 2 + slot) * 2 * 128 * 128 + pcol + col] = v;
            epi_bar();  // the release store below publishes the whole CTA's writes
            if (lead_warp && lane == 0) flag_set(pflag + blockIdx.x * 2 + slot, c.epoch);
            continue;
        }
        if (split) v += later;
        if (kGateUp) {
            if (warp >= 6) up_s[col - 128] = v;
            epi_bar();
            if (warp < 6) {
                const float h = silu_mul(v, up_s[col]);
                const int ex = mxfp8_exponent(warp_max(fabsf(h)));
                const uint32_t code = f32x2_to_e4m3x2(scale_pow2(h, ex), 0.f) & 0xFFu;
                a.hq[(size_t)s * a.I + f0 + col] = (uint8_t)code;
                // h's scale rows in the layout of the A scale copies: per K
                // step of the down GEMM 16 bytes, block kk once per lane quarter
                const int blk = (f0 + col - lane) / 32;
                if (lane < 4) a.hs[((size_t)s * (a.I / 128) + blk / 4) * 16 + 4 * lane + blk % 4] = (uint8_t)(ex + 127);
            }
            epi_bar();
            if (lead_warp && lane == 0) flag_set(a.h_flag + gt, c.epoch);
        } else if (s < c.k - 1) {
            word_set(a.yw + (size_t)gt * 256 + col, ((unsigned long long)c.epoch << 32) | __float_as_uint(v));
        } else {
            // the last expert's tile of block m: combine the block in
            // ascending expert order, this tile's y from registers, the
            // others' from their epoch-tagged words (all loads in flight
            // at once; a word of an earlier launch is polled again)
            unsigned long long yv[kMaxTopK - 1];
            const unsigned long long* yp = a.yw + (size_t)m * 256 + col;  // expert ss: + ss * MT * 256
#pragma unroll
            for (int ss = 0; ss < kMaxTopK - 1; ++ss) yv[ss] = ss < c.k - 1 ? word_get(yp + (size_t)ss * MT * 256) : 0ull;
            const bool ok = words_wait(yp, (size_t)MT * 256, c.k - 1, c.epoch, c.abort_flag, a.wait_ns, yv);
            float o = 0.f;
#pragma unroll
            for (int ss = 0; ss < kMaxTopK - 1; ++ss)
                if (ss < c.k - 1) o += c.seg_w[ss] * __uint_as_float((uint32_t)yv[ss]);
            if (!ok) c.give_up(a);
            o += c.seg_w[c.k - 1] * v;
            a.out[f0 + col] = o;
        }
    }
}

// The routing weights of the decode token by one warp: lane j < k takes the
// j-th selection sel[j] (router order); w_j = w_scale * s_j / (s_0 + ... +
// s_{k-1}), s = sqrt(softplus(logit)) in fp32 (the arithmetic of
// route_token), then the tail pruning.  Returns the kept count m (0 when the
// token has no valid selection); lane j gets its expert and weight.
__device__ __forceinline__ int dec_weights(const DecArgs& a, const int* sel, const float* lg, int lane, int& e,
                                           float& wj) {
    const int k = a.k;
    e = lane < k ? sel[lane] : 0;
    const bool ok = __all_sync(0xFFFFFFFFu, e >= 0);
    float sv = 0.f;
    if (lane < k && ok) sv = sqrt_softplus(lg[e]);
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xFFFFFFFFu, sv, j));
    wj = (lane < k && ok) ? route_weight(a.w_scale, sv, sum) : 0.0f;
    if (!ok) return 0;
    return prunes(a.prune, k) ? prune_tail(wj, k, a.prune, lane) : k;
}

__global__ void __launch_bounds__(kTcThreads, 1)
k_decode(const __grid_constant__ CUtensorMap tmGU, const __grid_constant__ CUtensorMap tmDN, const DecArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecBarOff);
    uint32_t* words = reinterpret_cast<uint32_t*>(bars + 2 * kDecStages + 2 + kDecGroups);
    // words: [0] tmem base, [1] abort, [2] epoch, [3] routed, [4..7] spare,
    // then seg_e, seg_j, seg_w, sel, prod_e (8 each)
    int* seg_e = reinterpret_cast<int*>(words + 8);
    int* seg_j = seg_e + 8;
    float* seg_w = reinterpret_cast<float*>(seg_j + 8);
    int* sel = reinterpret_cast<int*>(seg_w + 8);
    int* prod_e = sel + 8;  // [8] the producer warp's own copy of seg_e
    float* lg = reinterpret_cast<float*>(smem + kDecFrontOff);  // the logits (E <= 1024)
    DecCtx c;
    c.smem = smem;
    c.bar0 = smem_u32(bars);
    c.abort_flag = reinterpret_cast<volatile int*>(words + 1);
    c.seg_e = seg_e;
    c.seg_j = seg_j;
    c.seg_w = seg_w;
    volatile int* routed_flag = reinterpret_cast<volatile int*>(words + 3);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = a.k, E = a.E;

    if (threadIdx.x == 0) {
        for (int st = 0; st < kDecStages; ++st) {
            mbar_init(c.full_bar(st), 1);
            mbar_init(c.empty_bar(st), 1);
        }
        mbar_init(c.tmem_full(), 1);
        mbar_init(c.tmem_empty(), kEpiWarps);
        for (int g = 0; g < kDecGroups; ++g) mbar_init(c.h_bar(g), 1);
        *c.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmGU);
        prefetch_tmap(&tmDN);
    }
    if (threadIdx.x < 8) sel[threadIdx.x] = -1;
    if (warp == 1) tmem_alloc(smem_u32(words), 512);
    // zero the x row and its scale rows (the h rows arrive whole)
    for (int i = threadIdx.x; i < (4096 + 512) / 16; i += kTcThreads)
        reinterpret_cast<uint4*>(smem + kDecXOff)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < kDecXScaleBytes / 16; i += kTcThreads)
        reinterpret_cast<uint4*>(smem + kDecTokScaleOff)[i] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = words[0];
    // trace: [0] entry, [8] wait end, [9] routed, [1] exit (thread 0)
    unsigned long long* trc = a.trace ? a.trace + (size_t)blockIdx.x * 12 : nullptr;
    if (trc && threadIdx.x == 0) trc[0] = globaltimer();
    pdl_launch_dependents();
    pdl_wait();
    if (trc && threadIdx.x == 0) trc[8] = globaltimer();

    // ---- the launch's epoch (used after the front); x loads in flight while
    // the logits are ranked
    unsigned long long n_launch = 0;
    if (threadIdx.x == 32) {
        // the launch counter: read here by every CTA (the previous launch,
        // which advanced it, has completed), advanced once at this launch's end
        n_launch = *reinterpret_cast<volatile unsigned long long*>(a.launches);
    }
    // x is loaded (and later quantised) by warps 1-9 alone: chunk (tid - 32)
    // + 288 r, so each warp holds 32 consecutive 8-element chunks
    const int nch = a.H / 8;  // 8-element chunks; a 32-block is 4 chunks of 4 aligned lanes
    constexpr int kXThreads = kTcThreads - 32;
    static_assert(2 * kXThreads >= 4096 / 8, "two rounds of chunks cover H <= 4096");
    // (x in host memory: CTA 0 alone reads it, the others take its device copy
    // later -- x is first needed by the MMAs, well after the routing)
    const bool x_staged = a.x_stage != nullptr;
    uint4 xr[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (warp > 0 && (!x_staged || blockIdx.x == 0)) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int ch = threadIdx.x - 32 + r * kXThreads;
            if (ch < nch) xr[r] = *reinterpret_cast<const uint4*>(a.x + (size_t)ch * 8);
        }
    }
    // top-k by rank (larger logit first, equal logits by lower index; NaN
    // never selected), in two rounds: each warp ranks a 32-logit chunk among
    // itself and keeps its local top k as candidates -- every global top-k
    // logit is one -- then thread t ranks candidate t among all candidates.
    const int nchunk = (E + 31) / 32;
    const int nc = nchunk * k;                             // <= 256
    int* ci = reinterpret_cast<int*>(smem + kDecFrontOff + 4096);   // candidate experts (-1: none)
    float* cv = reinterpret_cast<float*>(smem + kDecFrontOff + 5120);  // their logits (NaN: none)
    for (int chk = warp; chk < nchunk; chk += kTcThreads / 32) {
        const int e = chk * 32 + lane;
        const float v = e < E ? __ldg(a.logits + e) : __int_as_float(0x7FC00000);
        if (e < E) lg[e] = v;
        int r = 0;
#pragma unroll
        for (int l2 = 0; l2 < 32; ++l2) {
            const float u = __shfl_sync(0xFFFFFFFFu, v, l2);
            r += (u > v || (u == v && l2 < lane)) ? 1 : 0;
        }
        if (lane < k) {
            ci[chk * k + lane] = -1;
            cv[chk * k + lane] = __int_as_float(0x7FC00000);
        }
        __syncwarp();
        if (v == v && r < k) {
            ci[chk * k + r] = e;
            cv[chk * k + r] = v;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < nc; t += kTcThreads) {
        const int e = ci[t];
        if (e < 0) continue;
        const float v = cv[t];
        int r = 0;
#pragma unroll 8
        for (int t2 = 0; t2 < nc; ++t2) {  // empty slots hold NaN: never counted
            const float u = cv[t2];
            r += (int)(u > v) | ((int)(u == v) & (int)(ci[t2] < e));
        }
        if (r < k) sel[r] = e;
    }
    if (threadIdx.x == 32) words[2] = (uint32_t)n_launch + 1u;  // this launch's flag value
    __syncthreads();
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    if (warp == 0) {
        // the producer starts as soon as the experts are known, on its own
        // copy of them in ascending order (the other warps still finish the
        // routing weights)
        // (with a weight threshold it needs the weights to know the kept
        // experts: it computes them itself, as warp 2 does)
        int e = lane < k ? sel[lane] : 0;
        int m = __all_sync(0xFFFFFFFFu, e >= 0) ? k : 0;
        if (m > 0 && prunes(a.prune, k)) {
            if (a.prune.min_w > 0.f) {
                float wj;
                m = dec_weights(a, sel, lg, lane, e, wj);
            } else {
                m = a.prune.keep;  // the first `keep` of the router order
            }
        }
        if (m > 0) {
            int pos = 0;
            for (int j = 0; j < m; ++j) pos += (__shfl_sync(0xFFFFFFFFu, e, j) < e) ? 1 : 0;
            if (lane < m) prod_e[pos] = e;
            __syncwarp();
            DecCtx cp = c;
            cp.seg_e = prod_e;
            cp.epoch = words[2];
            cp.k = m;
            const int G = dec_groups(m);
            // it runs through all phases (the weights do not depend on h),
            // fetching each group's h once that group's first down weights
            // are on their way
            bool ok = true;
            for (int g = 0; g < G && ok; ++g)
                ok = dec_produce<true>(a, cp, &tmGU, dec_phase(m, false, g), g, stage, phase, lane);
            for (int g = 0; g < G && ok; ++g)
                ok = dec_produce<false>(a, cp, &tmDN, dec_phase(m, true, g), g, stage, phase, lane);
        }
    } else {
        if (x_staged) {
            if (blockIdx.x == 0) {
                // publish the raw x: stores, the barrier over warps 1-9, one release
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int ch = threadIdx.x - 32 + r * kXThreads;
                    if (ch < nch) *reinterpret_cast<uint4*>(a.x_stage + (size_t)ch * 8) = xr[r];
                }
                work_bar();
                if (threadIdx.x == 32) flag_set(a.x_flag, words[2]);
            } else {
                if (threadIdx.x == 32 && !flag_wait(a.x_flag, words[2], c.abort_flag, a.wait_ns)) c.give_up(a);
                work_bar();  // the acquire above, then the whole of warps 1-9
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int ch = threadIdx.x - 32 + r * kXThreads;
                    if (ch < nch) xr[r] = __ldcg(reinterpret_cast<const uint4*>(a.x_stage + (size_t)ch * 8));
                }
            }
        }
        // ---- quantise x into the resident token row (MXFP8, 32-blocks),
        // while the producer streams the first weights
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int ch = threadIdx.x - 32 + r * kXThreads;
            if (ch - lane >= nch) continue;  // warp-uniform (nch is a multiple of 32)
            const uint32_t wv[4] = {xr[r].x, xr[r].y, xr[r].z, xr[r].w};
            float v[8];
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(wv[i] << 16);
                v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
            const int ex = mxfp8_exponent(amax);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                lo |= f32x2_to_e4m3x2(scale_pow2(v[2 * i], ex), scale_pow2(v[2 * i + 1], ex)) << (16 * i);
                hi |= f32x2_to_e4m3x2(scale_pow2(v[4 + 2 * i], ex), scale_pow2(v[5 + 2 * i], ex)) << (16 * i);
            }
            const int h = ch * 8, b = ch >> 2;
            *reinterpret_cast<uint2*>(smem + kDecXOff + h) = make_uint2(lo, hi);
            // the scale row of K step b / 4: block b % 4, once per lane quarter
            smem[kDecTokScaleOff + (b / 4) * 16 + 4 * (ch & 3) + (b % 4)] = (uint8_t)(ex + 127);
        }
        // the quantised row and scales were written through the generic proxy;
        // the MMAs read them through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (warp == 2) {
            int e;
            float wj;
            const int m = dec_weights(a, sel, lg, lane, e, wj);
            if (lane < k && blockIdx.x == 0) {
                a.ids_out[lane] = lane < m ? e : -1;  // pruned slots: -1, weight 0
                a.w_out[lane] = wj;
            }
            // position among the kept experts in ascending expert order (the
            // combine order; ids are distinct)
            int pos = 0;
            for (int j = 0; j < m; ++j) pos += (__shfl_sync(0xFFFFFFFFu, e, j) < e) ? 1 : 0;
            if (lane < m) {
                seg_e[pos] = e;
                seg_w[pos] = wj;
                seg_j[pos] = lane;
            }
            if (lane == 0) {
                if (m == 0 && blockIdx.x == 0) raise_flag(a.err, ERR_BAD_ID);
                *routed_flag = m;
            }
        }
        __syncwarp();
        work_bar();  // the routing of warps 1-9 (the producer is on its way)
        c.epoch = words[2];
        c.k = *routed_flag;
        if (trc && threadIdx.x == 32) trc[9] = globaltimer();
        if (c.k > 0) {
            const int G = dec_groups(c.k);
            bool ok = true;
            for (int g = 0; g < G; ++g) {
                const DecPhase ph = dec_phase(c.k, false, g);
                if (warp == 1) ok = ok && dec_mma<true>(a, c, ph, g, stage, phase, acc_phase, lane);
                else dec_epilogue<true>(a, c, ph, acc_phase);
            }
            for (int g = 0; g < G; ++g) {
                const DecPhase ph = dec_phase(c.k, true, g);
                if (warp == 1) ok = ok && !*c.abort_flag && dec_mma<false>(a, c, ph, g, stage, phase, acc_phase, lane);
                else dec_epilogue<false>(a, c, ph, acc_phase);
            }
        } else {
            // no valid routing (ERR_BAD_ID is raised): every row is dropped,
            // as in the grouped path, and the output is zero
            for (int i = blockIdx.x * (kTcThreads - 32) + threadIdx.x - 32; i < a.H; i += gridDim.x * (kTcThreads - 32))
                a.out[i] = 0.f;
        }
    }
    __syncwarp();  // the producer / MMA lane rejoins its warp before the CTA barrier
    __syncthreads();
    if (trc && threadIdx.x == 0) trc[1] = globaltimer();
    // the next launch reads the counter only after this grid has completed
    if (blockIdx.x == 0 && threadIdx.x == 32) *a.launches = n_launch + 1ull;
    if (*c.abort_flag) spin_ns(200000);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(c.tmem, 512);
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
    // the block-scaled MMAs take UE8M0 scales per 32 elements: NVFP4 experts
    // (e4m3 scales per 16) run on the CUDA-core kernels
    if (L->cfg.weight_format != MOE_WEIGHTS_MXFP4) return cudaSuccess;
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
    cudaError_t e = cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
    if (e == cudaSuccess) e = set_smem_attr<true, kFmtE2M1>();
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
    g.wait_ns = L->wait_ns;
    g.a_tx = kFp4BoxTx;
    g.sk_part = L->sk_partials;
    g.sk_cnt = L->sk_counters;
    g.trace = L->trace;
    cudaError_t e = tc_launch<true, kFmtE2M1>(L, st->gu, st->xq, g, s);
    if (e == cudaSuccess && mid) e = record_stage(mid, s);
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
    d.trace = L->trace ? L->trace + (size_t)L->num_sms * 12 : nullptr;
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
    sg.trace = L->trace ? L->trace + (size_t)2 * L->num_sms * 12 : nullptr;
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
    sd.trace = L->trace ? L->trace + (size_t)3 * L->num_sms * 12 : nullptr;
    return tc_launch<false, kFmtE4M3>(L, st->sh_down, st->hq_sh, sd, s);
}

}  // namespace moe

namespace moe {

bool decode_supported(const moe_layer* L) {
    // x resident as H / 128 B tiles of 2 KB (64 KB), h of two experts as
    // I / 128 tiles each (2 x 32 KB); a CTA range spans at most two experts
    // when k * (H / 256) <= 2 * SMs (always so when split)
    const moe_config& c = L->cfg;
    return L->tc != nullptr && !c.has_shared && c.hidden % 256 == 0 && c.hidden <= 4096 &&
           c.inter <= 2048 && c.top_k <= kMaxTopK && c.top_k * (c.hidden / 256) <= 2 * L->num_sms;
}

// One token: route + layer in the cooperative decode kernel.
cudaError_t launch_decode(moe_layer* L, const float* logits, const uint16_t* x, int32_t* ids, float* w,
                          float* out, cudaStream_t s, bool x_in_host) {
    const TcState* st = static_cast<const TcState*>(L->tc);
    DecArgs a{};
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
    a.gu_sf = L->gu_sf;
    a.down_sf = L->down_sf;
    a.hq = L->hq;
    a.hs = L->hs;
    a.yw = L->dec_yw;
    a.sk_part = L->sk_partials;
    int32_t* dw = L->sk_counters + kSkZeroed(L);
    a.launches = reinterpret_cast<unsigned long long*>(dw);
    a.piece_flag = reinterpret_cast<uint32_t*>(dw + 2);
    a.h_flag = a.piece_flag + 8 * L->num_sms;
    a.x_flag = a.h_flag + kDecMaxTiles;
    a.x_stage = x_in_host ? L->x_stage : nullptr;
    a.err = L->d_err;
    a.wait_ns = L->wait_ns;
    a.stall_h = L->stall_next_decode;
    L->stall_next_decode = 0;  // one-shot
    a.trace = L->trace;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L->num_sms);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kDecSmem;
    cfg.stream = s;
    // cooperative (all CTAs co-resident for the waits on each other's flags) and
    // programmatic dependent launch: a CTA takes its SM as soon as the
    // previous kernel's CTA there exits, runs its prologue and waits in
    // griddepcontrol.wait for that kernel's completion
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    L->launches += 1;
    return cudaLaunchKernelEx(&cfg, k_decode, st->gu, st->down, a);
}

}  // namespace moe
