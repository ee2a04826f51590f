// route.cuh -- routing of one token by one warp (learned sqrt-softplus
// router), shared by the routing kernels and the whole-layer decode kernel.
#pragma once

#include <climits>
#include <cmath>

#include "common.cuh"

namespace moe {

// Tail pruning of a learned routing (guide, section 3.2 item 3: top-k below
// the layer's k and the adaptive tail, with variance-preserving rescaling;
// RFC on CPU kernels, item 5).  keep >= k and min_w <= 0 prune nothing.
struct RoutePrune {
    int keep;     // at most this many experts are kept
    float min_w;  // an expert after the first is kept only while its weight is >= min_w
    float rho;    // assumed pairwise correlation of expert outputs, [0, 1]
};

__device__ __forceinline__ bool prunes(const RoutePrune& p, int k) { return p.keep < k || p.min_w > 0.f; }

// The routing arithmetic is written with explicit round-to-nearest
// operations, so that no call site contracts a product and a sum into one
// fused operation: every kernel that routes a token (the routing kernels and
// the whole-layer decode kernel) gets the same fp32 bits.
// s = sqrt(softplus(l)), softplus(l) = max(l, 0) + log1p(exp(-|l|)).
__device__ __forceinline__ float sqrt_softplus(float l) {
    return __fsqrt_rn(__fadd_rn(fmaxf(l, 0.f), log1pf(expf(-fabsf(l)))));
}
// w = w_scale * s / sum
__device__ __forceinline__ float route_weight(float w_scale, float s, float sum) {
    return __fdiv_rn(__fmul_rn(w_scale, s), sum);
}

// Lane j < k holds w_j (router order, descending).  Expert 0 is kept, expert
// j >= 1 while j < keep and w_j >= min_w: the first that fails ends the kept
// prefix of length m (returned).  Kept weights are multiplied by
//   sqrt(((1 - rho) S2 + rho S1^2) / ((1 - rho) S2' + rho S1'^2)),
// S1, S2 = sum of w_j and of w_j^2 over all k, S1', S2' over the kept ones
// (rho = 0: L2 quadrature, rho = 1: linear); pruned lanes get 0.  Sums in
// ascending j, fp32.  Every lane of the warp calls it.
__device__ __forceinline__ int prune_tail(float& wj, int k, const RoutePrune& p, int lane) {
    const bool fail = lane >= 1 && lane < k && (lane >= p.keep || !(wj >= p.min_w));
    const unsigned fm = __ballot_sync(0xFFFFFFFFu, fail);
    const int m = fm ? __ffs(fm) - 1 : k;
    if (m < k) {
        float s1a = 0.f, s2a = 0.f, s1k = 0.f, s2k = 0.f;
        for (int j = 0; j < k; ++j) {
            const float v = __shfl_sync(0xFFFFFFFFu, wj, j);
            const float v2 = __fmul_rn(v, v);
            s1a = __fadd_rn(s1a, v);
            s2a = __fadd_rn(s2a, v2);
            if (j < m) {
                s1k = __fadd_rn(s1k, v);
                s2k = __fadd_rn(s2k, v2);
            }
        }
        const float r1 = __fsub_rn(1.f, p.rho);
        const float num = __fadd_rn(__fmul_rn(r1, s2a), __fmul_rn(p.rho, __fmul_rn(s1a, s1a)));
        const float den = __fadd_rn(__fmul_rn(r1, s2k), __fmul_rn(p.rho, __fmul_rn(s1k, s1k)));
        const float alpha = __fsqrt_rn(__fdiv_rn(num, den));
        wj = lane < m ? __fmul_rn(wj, alpha) : 0.f;
    }
    return m;
}

// ------------------------------------------------------------------ route --
// One warp per token.  The top-k by score s = sqrt(softplus(logit)) is the
// top-k by logit (s is strictly increasing), so the selection compares the
// fp32 logits exactly: k warp-wide argmax passes, equal values to the lower
// expert index (guide, section 1: SQRT_SOFTPLUS gating, top-k).  Lane j < k
// then evaluates s_j in fp32 and every lane sums s_0..s_{k-1} in that order;
// w_j = w_scale * s_j / sum (guide, section 3.2); then the tail pruning, if
// any (pruned slots: id -1, weight 0).
// Routing of one token by one warp: writes ids_t[0..k) and w_t[0..k).
// The k argmax passes of route_token over the lane's logits held in
// registers (kPer per lane: experts lane, lane + 32, ...; E <= 32 kPer).
template <int kPer>
__device__ __forceinline__ bool route_select(const float* __restrict__ row, int E, int k, int lane, int& my_sel,
                                             float& my_logit) {
    float lv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) lv[i] = lane + 32 * i < E ? __ldg(row + lane + 32 * i) : 0.f;
    uint32_t taken = 0;  // bit i <-> expert lane + 32 i
    bool ok = true;
    for (int j = 0; j < k; ++j) {
        float best = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane + 32 * i;
            if (e >= E || ((taken >> i) & 1u)) continue;
            const float v = lv[i];
            if (v > best || (v == best && e < bi)) { best = v; bi = e; }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
        }
        if (bi >= E) { ok = false; bi = -1; }
        if (lane == j) { my_sel = bi; my_logit = best; }
        if (bi >= 0 && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    return ok;
}

__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, float w_scale,
                            const RoutePrune& prune, int32_t* __restrict__ ids_t,
                            float* __restrict__ w_t, uint32_t* err, int lane) {
    int my_sel = -1;     // lane j keeps the j-th selection
    float my_logit = 0.f;
    const bool ok = E <= 256 ? route_select<8>(row, E, k, lane, my_sel, my_logit)
                             : route_select<32>(row, E, k, lane, my_sel, my_logit);
    float s = 0.f;
    if (lane < k && my_sel >= 0) s = sqrt_softplus(my_logit);
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xFFFFFFFFu, s, j));
    float wj = (lane < k && ok) ? route_weight(w_scale, s, sum) : 0.0f;
    int m = k;
    if (ok && prunes(prune, k)) m = prune_tail(wj, k, prune, lane);
    if (lane < k) {
        ids_t[lane] = (ok && lane < m) ? my_sel : -1;
        w_t[lane] = wj;
    }
    if (!ok && lane == 0) raise_flag(err, ERR_BAD_ID);
}

}  // namespace moe
