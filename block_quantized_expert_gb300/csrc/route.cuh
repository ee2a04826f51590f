// route.cuh -- routing of one token by one warp (learned sqrt-softplus
// router), shared by the routing kernels and the whole-layer decode kernel.
#pragma once

#include <climits>
#include <cmath>

#include "common.cuh"

namespace moe {

// ------------------------------------------------------------------ route --
// One warp per token.  The top-k by score s = sqrt(softplus(logit)) is the
// top-k by logit (s is strictly increasing), so the selection compares the
// fp32 logits exactly: k warp-wide argmax passes, equal values to the lower
// expert index (guide, section 1: SQRT_SOFTPLUS gating, top-k).  Lane j < k
// then evaluates s_j in fp32 and every lane sums s_0..s_{k-1} in that order;
// w_j = w_scale * s_j / sum (guide, section 3.2).
// Routing of one token by one warp: writes ids_t[0..k) and w_t[0..k).
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, float w_scale,
                            int32_t* __restrict__ ids_t, float* __restrict__ w_t, uint32_t* err,
                            int lane) {
    uint32_t taken = 0;  // bit i <-> expert lane + 32 i
    int my_sel = -1;     // lane j keeps the j-th selection
    float my_logit = 0.f;
    bool ok = true;
    for (int j = 0; j < k; ++j) {
        float best = -INFINITY;
        int bi = INT_MAX;
        for (int i = 0, e = lane; e < E; ++i, e += 32) {
            if ((taken >> i) & 1u) continue;
            float v = __ldg(row + e);
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
    float s = 0.f;
    if (lane < k && my_sel >= 0)
        s = sqrtf(fmaxf(my_logit, 0.f) + log1pf(expf(-fabsf(my_logit))));
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, s, j);
    if (lane < k) {
        ids_t[lane] = ok ? my_sel : -1;
        w_t[lane] = ok ? w_scale * s / sum : 0.0f;
    }
    if (!ok && lane == 0) raise_flag(err, ERR_BAD_ID);
}

}  // namespace moe
