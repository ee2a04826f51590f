/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle of the routed-expert FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls, links or includes
 * this file; only the tests, the smoke check and the bench's CPU-baseline
 * leg load it.  It shares no code, header, table or helper with the CUDA
 * path and never reads a value the CUDA path produced.
 *
 * What it computes (all arithmetic in double; every intermediate quantised
 * value is produced exactly as the format definition says):
 *
 *  - the layer, "DeepSeek-V4-Flash 284B - Deep-Dive Mathematical & Kernel
 *    Guide", section 3.2 (the FFN output equation): y = e_shared(x) +
 *    sum_i w_i e_{k_i}(x) with sum_i w_i = w_scale = 1.5 (section 1);
 *  - the router, same guide section 1: gating function sqrt(softplus(logit)),
 *    top-k over the routed experts, the k selected scores normalised to sum
 *    to w_scale; and the hash-routed layers: a token-id -> expert table
 *    (tid2eid) with flat weights (section 1; section 3.2 item 1);
 *  - the expert FFN, same guide section 4 (the SwiGLU equation):
 *    h_j = g_j / (1 + e^{-g_j}) * u_j with g = W_gate x, u = W_up x,
 *    y = W_down h;
 *  - the token -> expert grouping that MUL_MAT_ID performs (section 2,
 *    "row-group reuse" / "batched expert bucket aggregation"), here a stable
 *    counting sort of the rows t*k+j by expert;
 *  - the formats: routed experts are MXFP4, i.e. e2m1 elements in 32-element
 *    blocks with a UE8M0 (E8M0) scale (colibri "DeepSeek V4 target engine",
 *    intro: experts stay native fp4; CISM VALIDATION "4-bit scheme study",
 *    row "E2M1 + E8M0 b32 (OCP MXFP4)"); the dense shared expert is fp8
 *    e4m3 with UE8M0 block scales (colibri intro), one scale per 128x128
 *    tile; activations entering a matmul are MXFP8: e4m3 elements in
 *    32-element blocks with a UE8M0 scale (colibri "Linux CUDA tier": the
 *    MXFP8 path), scale 2^(floor(log2 amax) - 8), round to nearest even,
 *    saturating at +-448, sign kept (so -0 encodes 0x80);
 *  - the NVFP4-style variant of the routed experts (CISM VALIDATION "4-bit
 *    quantization scheme study", row "E2M1 + E4M3 b16 (NVFP4 granularity)"):
 *    e2m1 elements in 16-element blocks with an e4m3 block scale, and (the
 *    reading taken here, since an e4m3 scale alone cannot reach the small
 *    magnitudes of the weights) one fp32 scale per expert matrix:
 *    value = e2m1(code) * e4m3(block scale) * matrix scale.
 *
 * Readings where the pages are silent are listed in the design notes; the
 * ones that shape this code: the top-k is plain (one expert group), ties in
 * the score go to the lower expert index; the routing weight multiplies the
 * down-projection output (after requantisation of h); the routed experts of
 * a token are summed in ascending expert order, the shared expert last.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* formats                                                                  */
/* ------------------------------------------------------------------------ */

/* e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/NaN.          */
double orc_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* e4m3 (fn variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * S.1111.111 is NaN, no infinities, max finite 448.                        */
double orc_e4m3_value(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);            /* subnormal: m/8 * 2^-6 */
    else        mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* UE8M0: unsigned power of two 2^(c - 127); 0xff is NaN.                  */
double orc_ue8m0_value(int code) {
    if (code == 255) return NAN;
    return ldexp(1.0, code - 127);
}

/* Nearest e4m3 value to y, ties to the even code (= even mantissa bit);
 * magnitudes above the largest finite value saturate to 448; the sign of y
 * is kept, also when the magnitude rounds to zero.  y must not be NaN.     */
int orc_e4m3_encode(double y) {
    int neg = signbit(y) ? 1 : 0;
    double mag = fabs(y);
    int c;
    if (mag >= 448.0) {
        c = 126;
    } else {
        /* largest code lo with value(lo) <= mag, by bisection over 0..126  */
        int lo = 0, hi = 126;
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (orc_e4m3_value(mid) <= mag) lo = mid; else hi = mid;
        }
        if (orc_e4m3_value(hi) <= mag) lo = hi;
        if (lo == 126) {
            c = 126;
        } else {
            double dlo = mag - orc_e4m3_value(lo), dhi = orc_e4m3_value(lo + 1) - mag;
            if (dlo < dhi) c = lo;
            else if (dhi < dlo) c = lo + 1;
            else c = (lo % 2 == 0) ? lo : lo + 1;
        }
    }
    return c | (neg << 7);
}

/* MXFP8 quantisation of n values (n a multiple of 32): per 32-block,
 * X = 2^(floor(log2 amax) - 8) (exponent clamped to [-127, 127]; a block of
 * zeros gets exponent -127), q = e4m3(v / X), s = UE8M0 byte of X.        */
void orc_mxfp8_quantize(const double* v, int n, uint8_t* q, uint8_t* s) {
    for (int b = 0; b < n / 32; ++b) {
        const double* blk = v + 32 * b;
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) if (fabs(blk[i]) > amax) amax = fabs(blk[i]);
        int ex;
        if (amax == 0.0) {
            ex = -127;
        } else {
            int e2;
            frexp(amax, &e2);          /* amax = f * 2^e2, f in [0.5, 1)   */
            ex = (e2 - 1) - 8;         /* floor(log2 amax) - 8             */
        }
        if (ex < -127) ex = -127;
        if (ex > 127) ex = 127;
        for (int i = 0; i < 32; ++i) q[32 * b + i] = (uint8_t)orc_e4m3_encode(ldexp(blk[i], -ex));
        s[b] = (uint8_t)(ex + 127);
    }
}

/* bf16 bits -> double (exact).                                             */
double orc_bf16_value(uint16_t bits) {
    union { uint32_t u; float f; } c;
    c.u = (uint32_t)bits << 16;
    return (double)c.f;
}

/* MXFP8 quantisation of T bf16 rows of length H: q [T][H], s [T][H/32].   */
int orc_quantize_bf16(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s) {
    if (H % 32) return 1;
    double* row = (double*)malloc(sizeof(double) * (size_t)H);
    if (!row) return 2;
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) row[h] = orc_bf16_value(x[(size_t)t * H + h]);
        orc_mxfp8_quantize(row, H, q + (size_t)t * H, s + (size_t)t * (H / 32));
    }
    free(row);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* routing                                                                  */
/* ------------------------------------------------------------------------ */

double orc_softplus(double l) { return (l > 0 ? l : 0.0) + log1p(exp(-fabs(l))); }
double orc_sqrt_softplus(double l) { return sqrt(orc_softplus(l)); }

/* Learned router: s_e = sqrt(softplus(logit_e)); the k largest scores, in
 * descending order, ties to the lower index; w_j = w_scale * s_j / sum s.  */
int orc_route_learned(const float* logits, int T, int E, int k, double w_scale,
                      int32_t* ids, double* w) {
    if (k < 1 || k > E) return 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
    if (!s || !taken) { free(s); free(taken); return 2; }
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) s[e] = orc_sqrt_softplus((double)logits[(size_t)t * E + e]);
        memset(taken, 0, (size_t)E);
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || s[e] > s[best])) best = e;
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
            sum += s[best];
        }
        for (int j = 0; j < k; ++j)
            w[(size_t)t * k + j] = w_scale * s[ids[(size_t)t * k + j]] / sum;
    }
    free(s);
    free(taken);
    return 0;
}

/* Tail pruning of a learned routing with variance-preserving rescaling
 * (guide, section 3.2 item 3: top-k below 6 and the adaptive tail with
 * L2-quadrature rescaling, and the general factor alpha_gen(rho); RFC on CPU
 * kernels, item 5: adaptive pruning below a weight threshold).
 *
 * For each token, in router order (descending score): expert 0 is kept;
 * expert j >= 1 is kept while j < keep and w_j >= min_w -- the first one that
 * fails ends the kept prefix of length m.  With
 *   A = (1 - rho) * sum_{j<k} w_j^2 + rho * (sum_{j<k} w_j)^2,
 *   B = (1 - rho) * sum_{j<m} w_j^2 + rho * (sum_{j<m} w_j)^2,
 * the kept weights become sqrt(A / B) * w_j (rho = 0: the L2 factor, which
 * keeps the sum of squares; rho = 1: the linear L1 factor, which keeps the
 * sum); the pruned slots become id -1, weight 0.  In place on [T][k].      */
int orc_route_prune(int32_t* ids, double* w, int T, int k, int keep, double min_w, double rho) {
    if (k < 1 || keep < 1 || !(rho >= 0.0 && rho <= 1.0)) return 1;
    for (int t = 0; t < T; ++t) {
        int32_t* id = ids + (size_t)t * k;
        double* wt = w + (size_t)t * k;
        int m = 1;
        while (m < k && m < keep && wt[m] >= min_w) ++m;
        if (m == k) continue;
        double s1a = 0.0, s2a = 0.0, s1k = 0.0, s2k = 0.0;
        for (int j = 0; j < k; ++j) {
            s1a += wt[j];
            s2a += wt[j] * wt[j];
            if (j < m) {
                s1k += wt[j];
                s2k += wt[j] * wt[j];
            }
        }
        double alpha = sqrt(((1.0 - rho) * s2a + rho * s1a * s1a) / ((1.0 - rho) * s2k + rho * s1k * s1k));
        for (int j = 0; j < k; ++j) {
            if (j < m) {
                wt[j] *= alpha;
            } else {
                id[j] = -1;
                wt[j] = 0.0;
            }
        }
    }
    return 0;
}

/* Hash router: ids[t] = tid2eid[token_ids[t]] (table order), w = w_scale/k. */
int orc_route_hash(const int32_t* token_ids, int T, const int32_t* tid2eid, int V, int k,
                   double w_scale, int32_t* ids, double* w) {
    for (int t = 0; t < T; ++t) {
        int id = token_ids[t];
        if (id < 0 || id >= V) return 1;
        for (int j = 0; j < k; ++j) {
            ids[(size_t)t * k + j] = tid2eid[(size_t)id * k + j];
            w[(size_t)t * k + j] = w_scale / k;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* permutation                                                              */
/* ------------------------------------------------------------------------ */

/* Stable counting sort of the rows r = t*k + j by expert ids[r]:
 * offsets[e] = number of rows with expert < e (offsets[E] = the number of
 * rows placed); row_src[p] = the row placed at position p; row_dst[r] = its
 * position.  An id of -1 is an empty slot (a pruned expert): its row is not
 * placed and row_dst[r] = -1.                                              */
int orc_permute(const int32_t* ids, int T, int k, int E,
                int32_t* offsets, int32_t* row_src, int32_t* row_dst) {
    int R = T * k;
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int r = 0; r < R; ++r) {
        if (ids[r] == -1) continue;
        if (ids[r] < 0 || ids[r] >= E) return 1;
        offsets[ids[r] + 1] += 1;
    }
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    if (!cursor) return 2;
    for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int r = 0; r < R; ++r) {
        if (ids[r] == -1) {
            row_dst[r] = -1;
            continue;
        }
        int p = cursor[ids[r]]++;
        row_src[p] = r;
        row_dst[r] = p;
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* the layer                                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
    int H, I, E, k;
    /* routed experts, MXFP4: payload [E][rows][K/2] (even element in the low
     * nibble), scales [E][rows][K/32]; gate/up rows = I, K = H; down rows =
     * H, K = I.                                                           */
    const uint8_t *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
    /* shared expert (or all NULL): e4m3 [rows][K], UE8M0 [rows/128][K/128] */
    const uint8_t *sh_gate_q, *sh_gate_s, *sh_up_q, *sh_up_s, *sh_down_q, *sh_down_s;
    /* routed-expert weight format: 0 MXFP4 (above); 1 NVFP4-style: the same
     * payload, scales e4m3 [E][rows][K/16], and fp32 matrix scales [E]     */
    int wfmt;
    const float *gate_g, *up_g, *down_g;
} orc_layer;

/* Decode tables, filled once from the value functions above.               */
static double tab_e2m1[16], tab_e4m3[256], tab_ue8m0[256];
static int tables_ready = 0;

static void init_tables(void) {
    if (tables_ready) return;
    for (int c = 0; c < 16; ++c) tab_e2m1[c] = orc_e2m1_value(c);
    for (int c = 0; c < 256; ++c) { tab_e4m3[c] = orc_e4m3_value(c); tab_ue8m0[c] = orc_ue8m0_value(c); }
    tables_ready = 1;
}

/* Value of element (row, col) of an MXFP4 matrix with K columns.           */
static double mxfp4_at(const uint8_t* q, const uint8_t* s, int K, size_t row, int col) {
    uint8_t byte = q[row * (size_t)(K / 2) + (size_t)(col / 2)];
    int code = (col % 2 == 0) ? (byte & 15) : (byte >> 4);
    return tab_e2m1[code] * tab_ue8m0[s[row * (size_t)(K / 32) + (size_t)(col / 32)]];
}

/* NVFP4-style element: e2m1(code) * e4m3(block scale byte) * matrix scale. */
double orc_nvfp4_value(int code, int sbyte, double g) {
    return orc_e2m1_value(code) * orc_e4m3_value(sbyte) * g;
}

/* Value of element (row, col) of an NVFP4-style matrix with K columns and
 * matrix scale g.                                                           */
static double nvfp4_at(const uint8_t* q, const uint8_t* s, int K, size_t row, int col, double g) {
    uint8_t byte = q[row * (size_t)(K / 2) + (size_t)(col / 2)];
    int code = (col % 2 == 0) ? (byte & 15) : (byte >> 4);
    return tab_e2m1[code] * tab_e4m3[s[row * (size_t)(K / 16) + (size_t)(col / 16)]] * g;
}

/* Element (row, col) of routed expert e's matrix (K columns; row counted
 * from the expert's first row) in the layer's weight format.              */
static double routed_at(const orc_layer* L, const uint8_t* q, const uint8_t* s, const float* g, int K,
                        int e, int rows, int row, int col) {
    size_t r = (size_t)e * rows + row;
    return L->wfmt == 1 ? nvfp4_at(q, s, K, r, col, (double)g[e]) : mxfp4_at(q, s, K, r, col);
}

/* Value of element (row, col) of an fp8 matrix with 128x128 tile scales.   */
static double fp8_tile_at(const uint8_t* q, const uint8_t* s, int K, size_t row, int col) {
    double v = tab_e4m3[q[row * (size_t)K + (size_t)col]];
    return v * tab_ue8m0[s[(row / 128) * (size_t)(K / 128) + (size_t)(col / 128)]];
}

/* One SwiGLU expert on one dequantised MXFP8 row xd[H]; e < 0 selects the
 * shared expert.  Writes y[H] and the MXFP8 bytes of h (hq[I], hs[I/32]).  */
static void expert_ffn(const orc_layer* L, int e, const double* xd, double* hbuf,
                       uint8_t* hq, uint8_t* hs, double* y) {
    int H = L->H, I = L->I;
    for (int j = 0; j < I; ++j) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            double wg, wu;
            if (e >= 0) {
                wg = routed_at(L, L->gate_q, L->gate_s, L->gate_g, H, e, I, j, c);
                wu = routed_at(L, L->up_q, L->up_s, L->up_g, H, e, I, j, c);
            } else {
                wg = fp8_tile_at(L->sh_gate_q, L->sh_gate_s, H, (size_t)j, c);
                wu = fp8_tile_at(L->sh_up_q, L->sh_up_s, H, (size_t)j, c);
            }
            g += xd[c] * wg;
            u += xd[c] * wu;
        }
        hbuf[j] = g / (1.0 + exp(-g)) * u;
    }
    orc_mxfp8_quantize(hbuf, I, hq, hs);
    for (int j = 0; j < I; ++j) hbuf[j] = tab_e4m3[hq[j]] * tab_ue8m0[hs[j / 32]];
    for (int c = 0; c < H; ++c) {
        double acc = 0.0;
        for (int j = 0; j < I; ++j) {
            double wd = (e >= 0) ? routed_at(L, L->down_q, L->down_s, L->down_g, I, e, H, c, j)
                                 : fp8_tile_at(L->sh_down_q, L->sh_down_s, I, (size_t)c, j);
            acc += hbuf[j] * wd;
        }
        y[c] = acc;
    }
}

/* Forward of the tokens listed in tok[0..n) of a batch of T tokens:
 * out[i][H] = sum over the token's k routed experts in ascending expert
 * order of w * expert(x) (+ the shared expert, if present, unweighted); an
 * id of -1 is an empty slot (a pruned expert) and adds nothing.
 * hq_out [n][k][I] / hs_out [n][k][I/32] (optional) receive the MXFP8 bytes
 * of h for the routed experts, in the token's own (j) order (zero for an
 * empty slot).                                                             */
int orc_layer_forward(const orc_layer* L, const uint16_t* x, const int32_t* ids,
                      const double* w, int T, const int32_t* tok, int n, double* out,
                      uint8_t* hq_out, uint8_t* hs_out) {
    int H = L->H, I = L->I, k = L->k, E = L->E;
    if (H % 128 || I % 128 || k < 1 || k > 64) return 1;
    if (L->wfmt != 0 && (L->wfmt != 1 || !L->gate_g || !L->up_g || !L->down_g)) return 1;
    init_tables();
    for (int i = 0; i < n; ++i) {
        if (tok[i] < 0 || tok[i] >= T) return 1;
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)tok[i] * k + j];
            if (e != -1 && (e < 0 || e >= E)) return 1;
        }
    }
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i) {
        int t = tok[i];
        uint8_t* xq = (uint8_t*)malloc((size_t)H);
        uint8_t* xs = (uint8_t*)malloc((size_t)H / 32);
        uint8_t* hq = (uint8_t*)malloc((size_t)I);
        uint8_t* hs = (uint8_t*)malloc((size_t)I / 32);
        double* xd = (double*)malloc(sizeof(double) * (size_t)H);
        double* xr = (double*)malloc(sizeof(double) * (size_t)H);
        double* y = (double*)malloc(sizeof(double) * (size_t)H);
        double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
        if (!xq || !xs || !hq || !hs || !xd || !xr || !y || !hbuf) {
#pragma omp atomic write
            status = 2;
        } else {
            double* o = out + (size_t)i * H;
            for (int c = 0; c < H; ++c) { xr[c] = orc_bf16_value(x[(size_t)t * H + c]); o[c] = 0.0; }
            orc_mxfp8_quantize(xr, H, xq, xs);
            for (int c = 0; c < H; ++c) xd[c] = tab_e4m3[xq[c]] * tab_ue8m0[xs[c / 32]];
            /* the token's experts in ascending expert order (ties: j order) */
            int order[64];
            for (int j = 0; j < k; ++j) order[j] = j;
            for (int a = 1; a < k; ++a)
                for (int b = a; b > 0 && ids[(size_t)t * k + order[b - 1]] > ids[(size_t)t * k + order[b]]; --b) {
                    int tmp = order[b]; order[b] = order[b - 1]; order[b - 1] = tmp;
                }
            for (int a = 0; a < k; ++a) {
                int j = order[a];
                int e = ids[(size_t)t * k + j];
                if (e == -1) {
                    if (hq_out) memset(hq_out + ((size_t)i * k + j) * I, 0, (size_t)I);
                    if (hs_out) memset(hs_out + ((size_t)i * k + j) * (I / 32), 0, (size_t)I / 32);
                    continue;
                }
                expert_ffn(L, e, xd, hbuf, hq, hs, y);
                double wt = w[(size_t)t * k + j];
                for (int c = 0; c < H; ++c) o[c] += wt * y[c];
                if (hq_out) memcpy(hq_out + ((size_t)i * k + j) * I, hq, (size_t)I);
                if (hs_out) memcpy(hs_out + ((size_t)i * k + j) * (I / 32), hs, (size_t)I / 32);
            }
            if (L->sh_gate_q) {
                expert_ffn(L, -1, xd, hbuf, hq, hs, y);
                for (int c = 0; c < H; ++c) o[c] += y[c];
            }
        }
        free(xq); free(xs); free(hq); free(hs); free(xd); free(xr); free(y); free(hbuf);
    }
    return status;
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
