/*
 * moe_tail_oracle.c -- plain, slow CPU oracle of the MoE decode tail.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load this file's library.  It
 * shares no code with the CUDA path: the BF16 conversions, the sum-of-squares
 * tree and every loop below are written here from the pages' statement of the
 * method, not taken from the kernels.
 *
 * Sources (vLLM API pages):
 *  [MS]  "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.moe.tail":
 *        module docstring (EP finalize and expert-TP finalize formulas),
 *        _TpTailKernel (gains, warp_sum_of_squares, normalized, the route sum
 *        "each product rounded alone"), _TailReduceKernel (rank-order FP32 sum
 *        of the BF16 partials), BoundTail.run (b = 0 does nothing).
 *  [KT]  "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.tail_runtime":
 *        module docstring (latent partial all-reduce, RMS norm, 3584 -> 7168
 *        up-projection, shared shard added into the output row).
 *  [KS]  "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.shared":
 *        module docstring and SharedUmma.owned_h (gate/up partials summed in
 *        FP32, gate and up rounded to BF16, activation into BF16 h, down
 *        projection pushed as BF16 with -0 made +0).
 *
 * Arithmetic.  The finalize steps run in IEEE binary32 with one rounding per
 * operation (built with -ffp-contract=off: no fused multiply-add), because the
 * pages fix FP32 sums and BF16 roundings there.  The GEMM steps run in double:
 * the pages fix only "FP32 accumulate", not an order, so the oracle takes the
 * exact-as-possible value and the GPU is held to a tolerance.
 *
 * Readings where the pages leave a step open:
 *  - sum of squares: lane l of 256-column chunk c owns columns 256c+8l..+7 and
 *    adds their squares in column order from +0; the 32 lanes combine by an
 *    xor butterfly over offsets 1,2,4,8,16; chunk sums fold in chunk order
 *    from +0.  This is the page's warp_sum_of_squares with the CTA's warps
 *    folded in order and a single band (split = 1).  Columns past P count 0.
 *  - inverse RMS = 1 / sqrt(ss * (float)(1/P) + eps), IEEE division and
 *    square root (the page writes rsqrt without stating its precision, so
 *    the correctly rounded form is used).
 *  - weight_before_norm: the norm gains g = bf16 gamma + gain_center multiply
 *    x before the sum of squares; otherwise after the normalisation.  The
 *    route weight always multiplies the normalised value, then adds into the
 *    route sum as a separately rounded product.
 *  - every BF16 that leaves a step has -0 replaced by +0.
 *  - latent tail: the slot sum is rounded to BF16 before the norm; the norm
 *    has gain center 0, y = bf16((x * inv) * gamma).
 *  - shared expert activation: SiLU, silu(g) = g / (1 + exp(-g)).
 *
 * Every entry returns 0 on success, -1 when its sizes are refused and -2 when
 * a host allocation fails (nothing is written then).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- BF16 <-> binary32 / binary64 --------------------------------------- */

float oracle_f32_from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a binary32 to BF16, nearest, ties to even; NaN stays a (quiet) NaN. */
uint16_t oracle_bf16_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

/* Round a binary64 straight to BF16 (nearest, ties to even).  Rounding first
 * to binary32 *to odd* and then to BF16 to nearest gives the correctly rounded
 * result because binary32 carries 16 more significand bits than BF16 (Boldo and
 * Melquiond, "Emulation of FMA and correctly rounded sums: proved algorithms
 * using rounding to odd", IEEE Trans. Computers 2008). */
uint16_t oracle_bf16_from_f64(double d) {
    if (isnan(d)) return 0x7fc0u;
    float f = (float)d;
    if ((double)f != d) {
        if (fabs((double)f) > fabs(d)) f = nextafterf(f, 0.0f); /* toward zero */
        uint32_t u;
        memcpy(&u, &f, 4);
        u |= 1u; /* the odd one of the two neighbours */
        memcpy(&f, &u, 4);
    }
    return oracle_bf16_from_f32(f);
}

static uint16_t pz(uint16_t h) { return h == 0x8000u ? 0u : h; }

static float bf16_round(float f) { return oracle_f32_from_bf16(oracle_bf16_from_f32(f)); }

/* ---- sum of squares tree ------------------------------------------------ */

float oracle_sum_of_squares(const float* v, int P) {
    float ss = 0.0f;
    int chunks = (P + 255) / 256;
    for (int c = 0; c < chunks; ++c) {
        float a[32], nb[32];
        for (int l = 0; l < 32; ++l) {
            float acc = 0.0f;
            for (int i = 0; i < 8; ++i) {
                int col = 256 * c + 8 * l + i;
                float e = col < P ? v[col] : 0.0f;
                float sq = e * e;
                acc = acc + sq;
            }
            a[l] = acc;
        }
        for (int off = 1; off < 32; off <<= 1) {
            for (int l = 0; l < 32; ++l) nb[l] = a[l] + a[l ^ off];
            memcpy(a, nb, sizeof a);
        }
        ss = ss + a[0];
    }
    return ss;
}

static float inverse_rms(float ss, int P, float eps) {
    float rcp = (float)(1.0 / (double)P);
    float mean = ss * rcp;
    float den = mean + eps;
    return 1.0f / sqrtf(den);
}

/* The inverse RMS on its own, for the pins of its rounding steps. */
float oracle_inverse_rms(float ss, int P, float eps) { return inverse_rms(ss, P, eps); }

static float route_weight(const void* w, int w_is_bf16, int64_t i) {
    return w_is_bf16 ? oracle_f32_from_bf16(((const uint16_t*)w)[i]) : ((const float*)w)[i];
}

/* One route row x (FP32 values of BF16) normalised with gains g, weighted by
 * w and added into part, column by column ([MS] _TpTailKernel.normalized and
 * the products/route sum that follow it). */
static void add_normalised_route(const float* x, const float* g, int wbn, float eps, float w,
                                 int P, float* v, float* part) {
    for (int c = 0; c < P; ++c) v[c] = wbn ? x[c] * g[c] : x[c];
    float inv = inverse_rms(oracle_sum_of_squares(v, P), P, eps);
    for (int c = 0; c < P; ++c) {
        float n = wbn ? v[c] * inv : (x[c] * inv) * g[c];
        float p = n * w;
        part[c] = part[c] + p;
    }
}

/* ---- EP finalize ([MS] module docstring, expert parallelism) -------------
 * rows  : BF16 [tp][rows_per_slot][P]   slot s's GEMM2 rows
 * idx   : int32 [tp][b][K]              route (t,k)'s row in slot s; local iff
 *                                       0 <= idx < rows_per_slot
 * w     : [b][K] FP32 (or BF16 if w_is_bf16)
 * gamma : BF16 [P]
 * out   : BF16 [b][P]
 * Per token: partial_s = bf16(sum over local routes in order of w*norm(x));
 * out = bf16(sum over s in order of partial_s), FP32 sums from +0. */
int oracle_ep_finalize(const uint16_t* rows, int64_t rows_per_slot, const int32_t* idx,
                       const void* w, int w_is_bf16, const uint16_t* gamma, float gain_center,
                       float eps, int wbn, int b, int tp, int K, int P, uint16_t* out) {
    if (b < 0 || tp < 1 || K < 1 || P < 1) return -1;
    float* g = malloc(sizeof(float) * P);
    float* x = malloc(sizeof(float) * P);
    float* v = malloc(sizeof(float) * P);
    float* part = malloc(sizeof(float) * P);
    float* o = malloc(sizeof(float) * P);
    if (!g || !x || !v || !part || !o) {
        free(g); free(x); free(v); free(part); free(o);
        return -2;
    }
    for (int c = 0; c < P; ++c) g[c] = oracle_f32_from_bf16(gamma[c]) + gain_center;
    for (int t = 0; t < b; ++t) {
        for (int c = 0; c < P; ++c) o[c] = 0.0f;
        for (int s = 0; s < tp; ++s) {
            for (int c = 0; c < P; ++c) part[c] = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t j = idx[((int64_t)s * b + t) * K + k];
                if (j < 0 || (int64_t)j >= rows_per_slot) continue; /* not this slot's */
                const uint16_t* row = rows + ((int64_t)s * rows_per_slot + j) * P;
                for (int c = 0; c < P; ++c) x[c] = oracle_f32_from_bf16(row[c]);
                add_normalised_route(x, g, wbn, eps, route_weight(w, w_is_bf16, (int64_t)t * K + k),
                                     P, v, part);
            }
            for (int c = 0; c < P; ++c) o[c] = o[c] + bf16_round(part[c]);
        }
        for (int c = 0; c < P; ++c) out[(int64_t)t * P + c] = pz(oracle_bf16_from_f32(o[c]));
    }
    free(g); free(x); free(v); free(part); free(o);
    return 0;
}

/* ---- expert-TP finalize ([MS] module docstring, expert TP) ----------------
 * partials : BF16 [tp][num_rows][P]  slot s's K-partial of every route row
 * idx      : int32 [b][K]            route (t,k)'s row, the same in every slot
 * x_r = bf16(sum over s in order of partial_s[row]); out = bf16(sum over routes
 * in order of w * norm(x_r)), from +0.  A route whose row is outside [0, num_rows)
 * contributes nothing (the page predicates its loads off; a zero row would add
 * w * 0, the same bits for any finite w). */
int oracle_tp_finalize(const uint16_t* partials, int64_t num_rows, const int32_t* idx,
                       const void* w, int w_is_bf16, const uint16_t* gamma, float gain_center,
                       float eps, int wbn, int b, int tp, int K, int P, uint16_t* out) {
    if (b < 0 || tp < 1 || K < 1 || P < 1) return -1;
    float* g = malloc(sizeof(float) * P);
    float* x = malloc(sizeof(float) * P);
    float* v = malloc(sizeof(float) * P);
    float* acc = malloc(sizeof(float) * P);
    if (!g || !x || !v || !acc) {
        free(g); free(x); free(v); free(acc);
        return -2;
    }
    for (int c = 0; c < P; ++c) g[c] = oracle_f32_from_bf16(gamma[c]) + gain_center;
    for (int t = 0; t < b; ++t) {
        for (int c = 0; c < P; ++c) acc[c] = 0.0f;
        for (int k = 0; k < K; ++k) {
            int32_t j = idx[(int64_t)t * K + k];
            if (j < 0 || (int64_t)j >= num_rows) continue; /* no row: contributes nothing */
            for (int c = 0; c < P; ++c) {
                float sum = 0.0f;
                for (int s = 0; s < tp; ++s)
                    sum = sum + oracle_f32_from_bf16(partials[((int64_t)s * num_rows + j) * P + c]);
                x[c] = bf16_round(sum);
            }
            add_normalised_route(x, g, wbn, eps, route_weight(w, w_is_bf16, (int64_t)t * K + k), P,
                                 v, acc);
        }
        for (int c = 0; c < P; ++c) out[(int64_t)t * P + c] = pz(oracle_bf16_from_f32(acc[c]));
    }
    free(g); free(x); free(v); free(acc);
    return 0;
}

/* ---- latent tail: slot sum + RMS norm ([KT] module docstring) --------------
 * latent : BF16 [tp][b][L]; gamma BF16 [L]; y : BF16 [b][L]
 * x = bf16(sum over s in order of latent_s), y = bf16((x * inv) * gamma). */
int oracle_latent_norm(const uint16_t* latent, const uint16_t* gamma, float eps, int b, int tp,
                       int L, uint16_t* y) {
    if (b < 0 || tp < 1 || L < 1) return -1;
    float* x = malloc(sizeof(float) * L);
    if (!x) return -2;
    for (int t = 0; t < b; ++t) {
        for (int c = 0; c < L; ++c) {
            float sum = 0.0f;
            for (int s = 0; s < tp; ++s)
                sum = sum + oracle_f32_from_bf16(latent[((int64_t)s * b + t) * L + c]);
            x[c] = bf16_round(sum);
        }
        float inv = inverse_rms(oracle_sum_of_squares(x, L), L, eps);
        for (int c = 0; c < L; ++c) {
            float n = (x[c] * inv) * oracle_f32_from_bf16(gamma[c]);
            y[(int64_t)t * L + c] = pz(oracle_bf16_from_f32(n));
        }
    }
    free(x);
    return 0;
}

/* ---- latent tail: up-projection + shared partials ([KT]) -------------------
 * y : BF16 [b][L]; w_up : BF16 [H][L]; shared : BF16 [tp_s][b][H] or NULL
 * out[t][n] = bf16(sum_c y[t][c] * w_up[n][c] + sum_s shared[s][t][n]), double. */
int oracle_latent_up(const uint16_t* y, const uint16_t* w_up, const uint16_t* shared, int tp_s,
                     int b, int L, int H, uint16_t* out) {
    if (b < 0 || L < 1 || H < 1 || tp_s < 0) return -1;
    double* yd = malloc(sizeof(double) * L);
    if (!yd) return -2;
    for (int t = 0; t < b; ++t) {
        for (int c = 0; c < L; ++c) yd[c] = oracle_f32_from_bf16(y[(int64_t)t * L + c]);
        for (int n = 0; n < H; ++n) {
            const uint16_t* wr = w_up + (int64_t)n * L;
            double acc = 0.0;
            for (int c = 0; c < L; ++c) acc += yd[c] * (double)oracle_f32_from_bf16(wr[c]);
            if (shared)
                for (int s = 0; s < tp_s; ++s)
                    acc += (double)oracle_f32_from_bf16(shared[((int64_t)s * b + t) * H + n]);
            out[(int64_t)t * H + n] = pz(oracle_bf16_from_f64(acc));
        }
    }
    free(yd);
    return 0;
}

/* ---- shared expert down projection ([KS] SharedBase.push) ------------------
 * h : BF16 [b][I]; w_down : BF16 [H][I]; out : BF16 [b][H] (read too if accumulate)
 * d = h . w_down (double); out = bf16(out + bf16(d)) (accumulate) or bf16(d). */
int oracle_shared_down(const uint16_t* h, const uint16_t* w_down, int b, int H, int I, uint16_t* out,
                       int accumulate) {
    if (b < 0 || H < 1 || I < 1) return -1;
    double* hd = malloc(sizeof(double) * I);
    if (!hd) return -2;
    for (int t = 0; t < b; ++t) {
        for (int i = 0; i < I; ++i) hd[i] = oracle_f32_from_bf16(h[(int64_t)t * I + i]);
        for (int n = 0; n < H; ++n) {
            const uint16_t* dr = w_down + (int64_t)n * I;
            double acc = 0.0;
            for (int i = 0; i < I; ++i) acc += hd[i] * (double)oracle_f32_from_bf16(dr[i]);
            uint16_t db = pz(oracle_bf16_from_f64(acc));
            uint16_t* o = out + (int64_t)t * H + n;
            if (accumulate) {
                float sum = oracle_f32_from_bf16(*o) + oracle_f32_from_bf16(db);
                *o = pz(oracle_bf16_from_f32(sum));
            } else {
                *o = db;
            }
        }
    }
    free(hd);
    return 0;
}

/* ---- fused shared expert ([KS]) --------------------------------------------
 * x : BF16 [b][H]; w_gate, w_up : BF16 [I][H]; w_down : BF16 [H][I]
 * h (out) : BF16 [b][I]; out : BF16 [b][H] (read too if accumulate)
 * gate = bf16(x . w_gate), up = bf16(x . w_up), h = bf16(silu(gate) * up),
 * then the down projection above. */
int oracle_shared_expert(const uint16_t* x, const uint16_t* w_gate, const uint16_t* w_up,
                         const uint16_t* w_down, int b, int H, int I, uint16_t* h_out,
                         uint16_t* out, int accumulate) {
    if (b < 0 || H < 1 || I < 1 || !h_out) return -1;
    double* xd = malloc(sizeof(double) * H);
    if (!xd) return -2;
    for (int t = 0; t < b; ++t) {
        for (int c = 0; c < H; ++c) xd[c] = oracle_f32_from_bf16(x[(int64_t)t * H + c]);
        for (int i = 0; i < I; ++i) {
            const uint16_t* gr = w_gate + (int64_t)i * H;
            const uint16_t* ur = w_up + (int64_t)i * H;
            double ga = 0.0, ua = 0.0;
            for (int c = 0; c < H; ++c) {
                ga += xd[c] * (double)oracle_f32_from_bf16(gr[c]);
                ua += xd[c] * (double)oracle_f32_from_bf16(ur[c]);
            }
            double gate = oracle_f32_from_bf16(oracle_bf16_from_f64(ga));
            double up = oracle_f32_from_bf16(oracle_bf16_from_f64(ua));
            double silu = gate / (1.0 + exp(-gate));
            h_out[(int64_t)t * I + i] = pz(oracle_bf16_from_f64(silu * up));
        }
    }
    free(xd);
    return oracle_shared_down(h_out, w_down, b, H, I, out, accumulate);
}
