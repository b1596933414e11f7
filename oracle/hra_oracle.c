/*
 * hra_oracle.c -- plain, slow CPU oracle of the Higgs-Audio-style hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the benchmark's CPU-baseline /
 * reference arm load this file's library.  It shares no code, header or table with the CUDA
 * library and includes none of it.
 *
 * What it computes (each function cites its source):
 *   - batched prefill of a Qwen3-style decoder backbone (from position 0, or one chunk per
 *     sequence after the positions already in the cache): embedding lookup, RMSNorm, merged QKV
 *     projection, per-head q/k RMSNorm + rotate-half RoPE with the KV-cache write, causal GQA
 *     attention over the used keys, o-projection + residual, RMSNorm, SwiGLU MLP + residual,
 *     final RMSNorm at the last used position ("Stabilize Higgs Audio termination and prefill",
 *     Summary; "flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its description and its
 *     per-layer chain);
 *   - the single-token decode pass through the same layers, fed an embedding;
 *   - the per-frame delayed-codebook step: audio-head logits, per-codebook argmax under the delay
 *     pattern with BOS/EOC handling and stop flags, and the sum of the K codebook embeddings
 *     ("Stabilize Higgs Audio termination and prefill", Summary and Root cause);
 *   - the same step with each codebook sampled (temperature, top-k, top-p, exponential race on
 *     per-row seeded Philox4x32-10 noise; vLLM-Omni PR #8226, Purpose and Test Plan);
 *   - the static-FP8 variant of the prefill projections (E4M3 weights with per-tensor scales,
 *     inputs quantized with calibrated static scales) and that calibration (the fp8_chain page,
 *     its description; "Stabilize Higgs Audio termination and prefill", Summary);
 *   - the NVFP4 codec and block-scaled linear of the chain's FP4 band (E2M1 elements, one E4M3
 *     scale per 16-element block, one fp32 global scale; the fp8_chain page, its precision bands).
 *
 * Arithmetic: fp32 on bf16-rounded weights and activations.  Values are rounded to bf16
 * (round-to-nearest-even) at these points and nowhere else: every RMSNorm output, the QKV
 * projection output, q and k after norm+RoPE (the norm stays fp32 into RoPE), the attention
 * output, gate and up projection outputs, the SwiGLU product, the residual after each add
 * (one rounding of r + acc), the final hidden, and the next-input embedding sum.  Logits stay
 * fp32.  Attention probabilities are exact fp32 (not rounded).  Dot products are summed in
 * ascending index order; compiled with -ffp-contract=off so x86 and Arm builds agree bit for bit.
 *
 * Readings where the pages are silent (stated once here, used throughout):
 *   - RMSNorm: y = bf16((x * (1/sqrt(ss/n + eps))) * g), one rounding, with ss the correctly
 *     rounded fp32 sum of squares (so the result does not hinge on a reduction order);
 *   - q/k norm gains are shared across heads ([head_dim]); GQA maps q head h to kv head
 *     h / (n_q / n_kv); attention scale 1/sqrt(head_dim); no biases;
 *   - RoPE pairs (i, i + hd/2), inv_freq_i = theta^(-2i/hd), positions restart at 0 in each
 *     sequence; cos/sin are evaluated in double and rounded to fp32;
 *   - delay pattern: codebook k lags k frames; see oracle_delay_step.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <limits.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    float rope_theta, rms_eps;
    int32_t n_codebooks, codebook_size, bos_id, eoc_id;
} oracle_dims;

typedef struct {
    const uint16_t *attn_norm, *w_qkv, *q_norm, *k_norm, *w_o, *mlp_norm, *w_gate_up, *w_down;
} oracle_layer;

/* ---------------------------------------------------------------- bf16 storage */

static float bf(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even; NaN stays NaN. */
static uint16_t to_bf(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void oracle_round_bf16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = to_bf(in[i]);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- RMSNorm */

/* y[r] = bf16((x[r] * (1/sqrt(ss/n + eps))) * g), ss = sum_squares(x[r]), per row of n.
 * Source: RMSNorm before each projection and the final norm (the fp8_chain page, its per-layer chain: the final
 * hidden is fin * rsqrt(mean(fin^2) + eps) * final_w). */
/* Sum of squares of n bf16 values as the fp32 rounding of the exact sum: each square of a bf16
 * value is exact in double and the double sum carries ~2^-53 relative error, so the result does not
 * depend on any summation order (the CUDA path reaches the same fp32 value by compensated
 * summation).  This is the mean of squares of RMSNorm evaluated once, correctly rounded. */
static float sum_squares(const uint16_t* x, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += (double)bf(x[i]) * (double)bf(x[i]);
    return (float)s;
}

void oracle_rmsnorm(const uint16_t* x, const uint16_t* g, int64_t rows, int n, float eps,
                    uint16_t* y) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * (int64_t)n;
        float ss = sum_squares(xr, n);
        float inv = 1.0f / sqrtf(ss / (float)n + eps);
        for (int i = 0; i < n; ++i) y[r * (int64_t)n + i] = to_bf((bf(xr[i]) * inv) * bf(g[i]));
    }
}

/* ---------------------------------------------------------------- linear */

/* y[t][j] = sum_k x[t][k] * w[j][k] in fp32, k ascending; w row-major [N][K] (out, in).
 * Each output is one plain sequential dot product (ascending k unless oracle_set_sum_order(1)).  The loop runs over output features j on the
 * outside and tokens t inside, so a weight row is read once per call whatever T is. */
static int g_sum_descending = 0;

/* Summation order of every dot product and sum whose order the method leaves open -- the linear
 * projections and attention's q.k, softmax-denominator and p.v sums: ascending (default) or
 * descending.  Both are plain evaluations of the same definition; running the oracle both ways
 * measures how far two correct bf16 evaluations of this model drift apart (the comparison floor
 * of any other implementation, whose fp32 sums take yet another order). */
void oracle_set_sum_order(int descending) { g_sum_descending = descending != 0; }

void oracle_linear(const uint16_t* x, const uint16_t* w, int T, int N, int K, float* y) {
    const int desc = g_sum_descending;
    float* xf = (float*)malloc(sizeof(float) * (size_t)T * (size_t)K);
    for (size_t i = 0; i < (size_t)T * (size_t)K; ++i) xf[i] = bf(x[i]);
    #pragma omp parallel
    {
        float* wrow = (float*)malloc(sizeof(float) * (size_t)K);
        #pragma omp for schedule(static)
        for (int j = 0; j < N; ++j) {
            for (int k = 0; k < K; ++k) wrow[k] = bf(w[(size_t)j * K + k]);
            for (int t = 0; t < T; ++t) {
                const float* xt = xf + (size_t)t * K;
                float acc = 0.0f;
                if (!desc)
                    for (int k = 0; k < K; ++k) acc += xt[k] * wrow[k];
                else
                    for (int k = K - 1; k >= 0; --k) acc += xt[k] * wrow[k];
                y[(size_t)t * N + j] = acc;
            }
        }
        free(wrow);
    }
    free(xf);
}

/* ---------------------------------------------------------------- RoPE */

/* cos/sin table [n_pos][hd/2]: angle = pos * theta^(-2i/hd), evaluated in double, rounded to fp32. */
void oracle_rope_table(int n_pos, int hd, double theta, float* cos_t, float* sin_t) {
    int half = hd / 2;
    for (int p = 0; p < n_pos; ++p)
        for (int i = 0; i < half; ++i) {
            double inv_freq = pow(theta, -(2.0 * (double)i) / (double)hd);
            double ang = (double)p * inv_freq;
            cos_t[p * half + i] = (float)cos(ang);
            sin_t[p * half + i] = (float)sin(ang);
        }
}

/* One head: RMSNorm over hd with gain g (kept fp32), then rotate-half RoPE at position pos,
 * rounded once to bf16.  Source: per-head q/k norm + RoPE before the cache write ("Stabilize Higgs
 * Audio termination and prefill", Summary: q/k norm, RoPE and the KV writes belong to the
 * kernelized prefill; the fp8_chain page: keys kept in host rotate-half layout in the cache). */
static void head_norm_rope(const uint16_t* x, const uint16_t* g, int hd, float eps,
                           const float* cos_p, const float* sin_p, uint16_t* out) {
    float xn[256];
    float ss = sum_squares(x, hd);
    float inv = 1.0f / sqrtf(ss / (float)hd + eps);
    for (int i = 0; i < hd; ++i) xn[i] = (bf(x[i]) * inv) * bf(g[i]);
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        float a = xn[i], b = xn[i + half], c = cos_p[i], s = sin_p[i];
        out[i] = to_bf(a * c - b * s);
        out[i + half] = to_bf(b * c + a * s);
    }
}

/* Batch form for tests: rows of x [rows][hd], positions pos[rows]. */
void oracle_qk_norm_rope(const uint16_t* x, const uint16_t* g, const int32_t* pos, int rows, int hd,
                         float eps, double theta, uint16_t* out) {
    int maxp = 0;
    for (int r = 0; r < rows; ++r) if (pos[r] > maxp) maxp = pos[r];
    float* ct = (float*)malloc(sizeof(float) * (size_t)(maxp + 1) * (hd / 2));
    float* st = (float*)malloc(sizeof(float) * (size_t)(maxp + 1) * (hd / 2));
    oracle_rope_table(maxp + 1, hd, theta, ct, st);
    for (int r = 0; r < rows; ++r)
        head_norm_rope(x + (size_t)r * hd, g, hd, eps, ct + (size_t)pos[r] * (hd / 2),
                       st + (size_t)pos[r] * (hd / 2), out + (size_t)r * hd);
    free(ct);
    free(st);
}

/* ---------------------------------------------------------------- attention */

/* Causal GQA attention of n rows at positions q_pos0 .. q_pos0+n-1 over the cache keys 0..pos.
 *   q   [n][nq][hd]   (post-RoPE, bf16)
 *   kc  [nkv][n_slots][hd], vc [nkv][n_slots][hd]   one sequence's cache for one layer
 *   out [n][nq*hd]    bf16(sum_j p_j v_j / sum_j p_j), p_j = exp(s_j - max s), s_j = q.k_j / sqrt(hd)
 *   probs (optional) [n][nq][n_keys_max]: the normalised probabilities (fp32), zeros past pos.
 * Source: dense attention over the used keys only, with trailing pads (the fp8_chain page, its
 * description and its mask check); causal because the backbone is a decoder. */
void oracle_attend(const uint16_t* q, const uint16_t* kc, const uint16_t* vc, int n_slots,
                   int q_pos0, int n, int nq, int nkv, int hd, uint16_t* out,
                   float* probs, int n_keys_max) {
    const float scale = 1.0f / sqrtf((float)hd);
    const int group = nq / nkv;
    #pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int i = 0; i < n; ++i) {
        for (int h = 0; h < nq; ++h) {
            int pos = q_pos0 + i;
            int kvh = h / group;
            const uint16_t* qi = q + ((size_t)i * nq + h) * hd;
            const uint16_t* kh = kc + (size_t)kvh * n_slots * hd;
            const uint16_t* vh = vc + (size_t)kvh * n_slots * hd;
            float* s = (float*)malloc(sizeof(float) * (size_t)(pos + 1));
            /* summation order of the three sums (q.k over the head dim, the softmax denominator
             * and p.v over the keys): ascending, or descending under oracle_set_sum_order(1) */
            const int desc = g_sum_descending;
            float m = -INFINITY;
            for (int j = 0; j <= pos; ++j) {
                float dot = 0.0f;
                for (int t = 0; t < hd; ++t) {
                    const int e = desc ? hd - 1 - t : t;
                    dot += bf(qi[e]) * bf(kh[(size_t)j * hd + e]);
                }
                s[j] = dot * scale;
                if (s[j] > m) m = s[j];
            }
            float l = 0.0f;
            for (int j = 0; j <= pos; ++j) s[j] = expf(s[j] - m);
            for (int t = 0; t <= pos; ++t) l += s[desc ? pos - t : t];
            for (int e = 0; e < hd; ++e) {
                float acc = 0.0f;
                for (int t = 0; t <= pos; ++t) {
                    const int j = desc ? pos - t : t;
                    acc += s[j] * bf(vh[(size_t)j * hd + e]);
                }
                out[(size_t)i * nq * hd + (size_t)h * hd + e] = to_bf(acc / l);
            }
            if (probs) {
                float* pr = probs + ((size_t)i * nq + h) * n_keys_max;
                for (int j = 0; j < n_keys_max; ++j) pr[j] = j <= pos ? s[j] / l : 0.0f;
            }
            free(s);
        }
    }
}

/* ---------------------------------------------------------------- FP8 (E4M3) variant */

/* OCP FP8 E4M3 ("fn": no infinities): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Normal codes (exponent field E > 0): (1 + M/8) * 2^(E-7); subnormals (E == 0): M/8 * 2^-6;
 * S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.  Encoding rounds to the
 * nearest code, ties to an even mantissa, and saturates finite overflow to +-448 (the satfinite
 * conversion); NaN stays NaN.  Source: the static-FP8 chain's E4M3 weights and activations
 * (the fp8_chain page, its description: RMSNorm then FP8, the FP8 GEMMs and the E4M3 maximum). */
float oracle_e4m3_decode(uint8_t c) {
    const int sgn = c >> 7, E = (c >> 3) & 15, M = c & 7;
    if (E == 15 && M == 7) return NAN;
    const double v = E == 0 ? (double)M / 8.0 * ldexp(1.0, -6) : (1.0 + (double)M / 8.0) * ldexp(1.0, E - 7);
    return (float)(sgn ? -v : v);
}

uint8_t oracle_e4m3_encode(float x) {
    if (x != x) return 0x7F;
    const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sgn | 0x7E;                 /* satfinite */
    /* quantum of the binade holding a (subnormal quantum below 2^-6) */
    int e = a > 0.0 ? (int)floor(log2(a)) : -6;
    if (e < -6) e = -6;
    const double q = ldexp(1.0, e - 3);
    double m = a / q;                                  /* exact: power-of-two scaling */
    double f = floor(m);
    const double frac = m - f;
    if (frac > 0.5 || (frac == 0.5 && fmod(f, 2.0) == 1.0)) f += 1.0;
    const double r = f * q;
    if (r >= 448.0) return sgn | 0x7E;
    if (r == 0.0) return sgn;
    if (r < ldexp(1.0, -6)) return sgn | (uint8_t)(r / ldexp(1.0, -9));   /* subnormal: M = r / 2^-9 */
    const int er = (int)floor(log2(r));
    const int M = (int)((r / ldexp(1.0, er) - 1.0) * 8.0);
    return sgn | (uint8_t)((er + 7) << 3) | (uint8_t)M;
}

/* out[i] = e4m3(bf(x[i]) / scale), the division in fp32. */
void oracle_quantize_e4m3(const uint16_t* x, int64_t n, float scale, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(bf(x[i]) / scale);
}

/* Per-tensor weight quantization: scale = max|w| / 448 (fp32; 1 when w is all zero), w8 = e4m3(w / scale). */
void oracle_quantize_weight_e4m3(const uint16_t* w, int64_t n, float* scale_out, uint8_t* out) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf(bf(w[i]));
        if (a > amax) amax = a;
    }
    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    *scale_out = scale;
    oracle_quantize_e4m3(w, n, scale, out);
}

/* y[t][j] = (sum_k x8[t][k] * w8[j][k]) * scale in fp32 (the products of two E4M3 values are exact
 * in fp32), k ascending (descending under oracle_set_sum_order(1)); w8 row-major [N][K]. */
void oracle_linear_fp8(const uint8_t* x8, const uint8_t* w8, int T, int N, int K, float scale, float* y) {
    const int desc = g_sum_descending;
    float lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = oracle_e4m3_decode((uint8_t)c);
    #pragma omp parallel for schedule(static)
    for (int j = 0; j < N; ++j) {
        const uint8_t* wr = w8 + (size_t)j * K;
        for (int t = 0; t < T; ++t) {
            const uint8_t* xr = x8 + (size_t)t * K;
            float s = 0.0f;
            for (int i = 0; i < K; ++i) {
                const int k = desc ? K - 1 - i : i;
                s += lut[xr[k]] * lut[wr[k]];
            }
            y[(size_t)t * N + j] = s * scale;
        }
    }
}

/* ---------------------------------------------------------------- NVFP4 (E2M1 + block scales) */

/* FP4 E2M1: 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit.  Exponent field 0 is
 * subnormal, m * 0.5; otherwise (1 + m/2) * 2^(e-1): the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 * No infinity or NaN.  Encoding rounds to the nearest value, ties to the even mantissa, and
 * saturates beyond 6 to +-6.  Source: the NVFP4 band of the prefill chain (the fp8_chain page, its precision
 * bands: the FFN pair and the output projection in NVFP4 with per-block scales); the element and
 * scale formats are NVIDIA's published NVFP4 definition, which the pages name but do not spell out. */
float oracle_e2m1_decode(uint8_t c) {
    const int sgn = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    const double v = e == 0 ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
    return (float)(sgn ? -v : v);
}

uint8_t oracle_e2m1_encode(float x) {
    const uint8_t sgn = signbit(x) ? 8 : 0;
    const double a = fabs((double)x);
    if (!(a < 6.0)) return sgn | 7;                    /* saturate (NaN too: the format has none) */
    /* candidates in code order; pick the nearest, a tie going to the even mantissa */
    int best = 0;
    double bd = a;
    for (int c = 1; c < 8; ++c) {
        const double d = fabs(a - (double)oracle_e2m1_decode((uint8_t)c));
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    return sgn | (uint8_t)best;
}

/* Global scale of an NVFP4 tensor: max|x| / (6 * 448) in fp32 (1 for an all-zero tensor), so that
 * every block scale fits E4M3. */
float oracle_nvfp4_global(const uint16_t* x, int64_t n) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf(bf(x[i]));
        if (a > amax) amax = a;
    }
    return amax > 0.0f ? amax / (6.0f * 448.0f) : 1.0f;
}

/* NVFP4 quantization of x [rows][K] (bf16), K a multiple of 16: each block of 16 consecutive
 * elements along K gets the E4M3 scale s_b = e4m3(amax_b / (6 g)) and the codes
 * e2m1(x / (g * dec(s_b))) (all 0 when dec(s_b) is 0); divisions in fp32.  codes: one code per
 * byte [rows][K]; scales [rows][K / 16]. */
void oracle_quantize_nvfp4(const uint16_t* x, int rows, int K, float g, uint8_t* codes, uint8_t* scales) {
    const int nb = K / 16;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const uint16_t* xb = x + (size_t)r * K + 16 * b;
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                const float a = fabsf(bf(xb[i]));
                if (a > amax) amax = a;
            }
            const uint8_t sc = oracle_e4m3_encode(amax / (6.0f * g));
            scales[(size_t)r * nb + b] = sc;
            const float step = g * oracle_e4m3_decode(sc);
            for (int i = 0; i < 16; ++i)
                codes[(size_t)r * K + 16 * b + i] = step > 0.0f ? oracle_e2m1_encode(bf(xb[i]) / step) : 0;
        }
}

/* y[t][j] = (g_a * g_w) * sum over blocks b (ascending; descending under oracle_set_sum_order(1))
 * of dec(sa[t][b]) * dec(sw[j][b]) * (sum over the block's 16 k ascending of e2m1(a) * e2m1(w)),
 * in fp32.  Each block's term is exact in fp32 (E2M1 products are multiples of 1/4 below 37, the
 * two E4M3 scales have 4-bit significands), so only the sum over blocks and the final scaling
 * round -- the order a block-scaled tensor-core MMA accumulates in. */
void oracle_linear_nvfp4(const uint8_t* a, const uint8_t* sa, const uint8_t* w, const uint8_t* sw, int T, int N,
                         int K, float g_a, float g_w, float* y) {
    const int desc = g_sum_descending;
    const int nb = K / 16;
    const float g = g_a * g_w;
    #pragma omp parallel for schedule(static)
    for (int j = 0; j < N; ++j)
        for (int t = 0; t < T; ++t) {
            float acc = 0.0f;
            for (int ib = 0; ib < nb; ++ib) {
                const int b = desc ? nb - 1 - ib : ib;
                float blk = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    const int k = 16 * b + i;
                    blk += oracle_e2m1_decode(a[(size_t)t * K + k]) * oracle_e2m1_decode(w[(size_t)j * K + k]);
                }
                acc += (oracle_e4m3_decode(sa[(size_t)t * nb + b]) * oracle_e4m3_decode(sw[(size_t)j * nb + b])) * blk;
            }
            y[(size_t)t * N + j] = acc * g;
        }
}

typedef struct {
    const uint8_t *w_qkv, *w_o, *w_gate_up, *w_down;   /* E4M3 weights, shapes as the bf16 ones */
    float w_scale[4];                                   /* qkv, o, gate_up, down */
    float a_scale[4];                                   /* static scale of each projection's input */
} oracle_fp8_layer;

/* NVFP4 band of the prefill chain (the fp8_chain page, its precision bands): the merged QKV stays
 * in static FP8, the output, gate/up and down projections run in NVFP4.
 *   w_qkv, w_scale[0], a_scale[0]      E4M3 QKV weights, their scale and the static input scale
 *   codes[p], scales[p] (p = 1, 2, 3)  E2M1 weight codes [N][K] (one per byte) and E4M3 block
 *                                      scales [N][K/16] of the output, gate/up and down weights
 *   w_scale[p], a_scale[p] (p >= 1)    the weights' fp32 global scale g_w, and the static fp32
 *                                      global scale g_a of the projection's input (its block scales
 *                                      are computed from each call's data) */
typedef struct {
    const uint8_t* w_qkv;
    const uint8_t* codes[4];
    const uint8_t* scales[4];
    float w_scale[4];
    float a_scale[4];
} oracle_nvfp4_layer;

/* One projection: bf16 (w8 == NULL and wc == NULL), FP8 (w8: the input quantized with the static
 * scale as, the result scaled by as * ws) or NVFP4 (wc / wsc: the input quantized to E2M1 codes with
 * per-16-element E4M3 block scales under the global scale as, then the block-scaled linear with
 * g_a = as, g_w = ws).  amax (optional) receives the max |input| seen. */
static void project(const uint16_t* x, const uint16_t* w, const uint8_t* w8, float ws, float as, int n, int N,
                    int K, float* y, float* amax, const uint8_t* wc, const uint8_t* wsc) {
    if (amax) {
        for (size_t i = 0; i < (size_t)n * K; ++i) {
            const float a = fabsf(bf(x[i]));
            if (a > *amax) *amax = a;
        }
    }
    if (wc != NULL) {
        uint8_t* xc = (uint8_t*)malloc((size_t)n * K);
        uint8_t* xs = (uint8_t*)malloc((size_t)n * (K / 16));
        oracle_quantize_nvfp4(x, n, K, as, xc, xs);
        oracle_linear_nvfp4(xc, xs, wc, wsc, n, N, K, as, ws, y);
        free(xc);
        free(xs);
        return;
    }
    if (w8 == NULL) {
        oracle_linear(x, w, n, N, K, y);
        return;
    }
    uint8_t* x8 = (uint8_t*)malloc((size_t)n * K);
    oracle_quantize_e4m3(x, (int64_t)n * K, as, x8);
    oracle_linear_fp8(x8, w8, n, N, K, as * ws, y);
    free(x8);
}

/* ---------------------------------------------------------------- decoder layers */

static float silu(float x) { return x / (1.0f + expf(-x)); }

/* Run n new rows of ONE sequence through every layer.
 *   x_in   [n][H] bf16 input embeddings of the new rows (positions start .. start+n-1)
 *   kv     this sequence's layer-0 cache block; layer l starts at kv + l * layer_stride;
 *          within a layer: K [nkv][n_slots][hd] then V [nkv][n_slots][hd]
 *   hidden [n][H] final-RMSNorm output of every new row (may be NULL)
 * Per layer (the fp8_chain page, its per-layer chain: norm -> QKV -> split/RoPE/cache -> attend -> o-proj, residual
 * add -> norm -> gate/up -> gated activation -> down, residual add; SwiGLU replaces that page's
 * GeGLU for the Qwen3-style backbone):
 *   y = RMSNorm(r; attn_norm); qkv = bf16(y W_qkv^T)
 *   q_h, k_j = bf16(RoPE(RMSNorm_hd(.; q_norm / k_norm), pos)); cache K[j][pos] = k_j, V[j][pos] = v_j
 *   a = attention(q, cache keys 0..pos);  r = bf16(r + a W_o^T)
 *   y = RMSNorm(r; mlp_norm); g = bf16(y W_gate^T), u = bf16(y W_up^T); h = bf16(silu(g) * u)
 *   r = bf16(r + h W_down^T) */
static void forward_rows(const oracle_dims* d, const oracle_layer* layers, const uint16_t* final_norm,
                         const uint16_t* x_in, int start, int n, uint16_t* kv, size_t layer_stride,
                         int n_slots, uint16_t* hidden, const oracle_fp8_layer* fp8, float* amax,
                         const oracle_nvfp4_layer* nv4) {
    const int H = d->hidden, nq = d->n_q_heads, nkv = d->n_kv_heads, hd = d->head_dim, F = d->ffn;
    const int Dq = nq * hd, Dqkv = (nq + 2 * nkv) * hd;
    const float eps = d->rms_eps;
    uint16_t* r = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * H);
    uint16_t* y = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * H);
    uint16_t* qkv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * Dqkv);
    uint16_t* qr = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * Dq);
    uint16_t* att = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * Dq);
    uint16_t* hmid = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * F);
    size_t fmax = (size_t)n * (size_t)(Dqkv > 2 * F ? Dqkv : 2 * F);
    if (fmax < (size_t)n * H) fmax = (size_t)n * H;
    float* acc = (float*)malloc(sizeof(float) * fmax);
    float* ct = (float*)malloc(sizeof(float) * (size_t)(start + n) * (hd / 2));
    float* st = (float*)malloc(sizeof(float) * (size_t)(start + n) * (hd / 2));
    oracle_rope_table(start + n, hd, (double)d->rope_theta, ct, st);
    memcpy(r, x_in, sizeof(uint16_t) * (size_t)n * H);

    for (int l = 0; l < d->n_layers; ++l) {
        const oracle_layer* L = &layers[l];
        uint16_t* kc = kv + (size_t)l * layer_stride;
        uint16_t* vc = kc + (size_t)nkv * n_slots * hd;
        /* attention block */
        oracle_rmsnorm(r, L->attn_norm, n, H, eps, y);
        /* the quantized projection p of layer l: FP8 (fp8, or the NVFP4 band's QKV) or NVFP4 */
#define PROJ_W8(p, fld) (fp8 ? fp8[l].fld : (nv4 && (p) == 0) ? nv4[l].w_qkv : NULL)
#define PROJ_WS(p) (fp8 ? fp8[l].w_scale[p] : nv4 ? nv4[l].w_scale[p] : 1.0f)
#define PROJ_AS(p) (fp8 ? fp8[l].a_scale[p] : nv4 ? nv4[l].a_scale[p] : 1.0f)
#define PROJ_WC(p) (nv4 && (p) > 0 ? nv4[l].codes[p] : NULL)
#define PROJ_WSC(p) (nv4 && (p) > 0 ? nv4[l].scales[p] : NULL)
        project(y, L->w_qkv, PROJ_W8(0, w_qkv), PROJ_WS(0), PROJ_AS(0), n, Dqkv, H, acc, amax ? amax + 4 * l : NULL,
                PROJ_WC(0), PROJ_WSC(0));
        for (size_t i = 0; i < (size_t)n * Dqkv; ++i) qkv[i] = to_bf(acc[i]);
        for (int i = 0; i < n; ++i) {
            int pos = start + i;
            const uint16_t* row = qkv + (size_t)i * Dqkv;
            const float* cp = ct + (size_t)pos * (hd / 2);
            const float* sp = st + (size_t)pos * (hd / 2);
            for (int h = 0; h < nq; ++h)
                head_norm_rope(row + (size_t)h * hd, L->q_norm, hd, eps, cp, sp,
                               qr + (size_t)i * Dq + (size_t)h * hd);
            for (int j = 0; j < nkv; ++j) {
                head_norm_rope(row + (size_t)(nq + j) * hd, L->k_norm, hd, eps, cp, sp,
                               kc + ((size_t)j * n_slots + pos) * hd);
                memcpy(vc + ((size_t)j * n_slots + pos) * hd, row + (size_t)(nq + nkv + j) * hd,
                       sizeof(uint16_t) * hd);
            }
        }
        oracle_attend(qr, kc, vc, n_slots, start, n, nq, nkv, hd, att, NULL, 0);
        project(att, L->w_o, PROJ_W8(1, w_o), PROJ_WS(1), PROJ_AS(1), n, H, Dq, acc, amax ? amax + 4 * l + 1 : NULL,
                PROJ_WC(1), PROJ_WSC(1));
        for (size_t i = 0; i < (size_t)n * H; ++i) r[i] = to_bf(bf(r[i]) + acc[i]);
        /* MLP block */
        oracle_rmsnorm(r, L->mlp_norm, n, H, eps, y);
        project(y, L->w_gate_up, PROJ_W8(2, w_gate_up), PROJ_WS(2), PROJ_AS(2), n, 2 * F, H, acc,
                amax ? amax + 4 * l + 2 : NULL, PROJ_WC(2), PROJ_WSC(2));
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < F; ++j) {
                float g = bf(to_bf(acc[(size_t)i * 2 * F + j]));
                float u = bf(to_bf(acc[(size_t)i * 2 * F + F + j]));
                hmid[(size_t)i * F + j] = to_bf(silu(g) * u);
            }
        project(hmid, L->w_down, PROJ_W8(3, w_down), PROJ_WS(3), PROJ_AS(3), n, H, F, acc,
                amax ? amax + 4 * l + 3 : NULL, PROJ_WC(3), PROJ_WSC(3));
#undef PROJ_W8
#undef PROJ_WS
#undef PROJ_AS
#undef PROJ_WC
#undef PROJ_WSC
        for (size_t i = 0; i < (size_t)n * H; ++i) r[i] = to_bf(bf(r[i]) + acc[i]);
    }
    if (hidden) oracle_rmsnorm(r, final_norm, n, H, eps, hidden);
    free(r); free(y); free(qkv); free(qr); free(att); free(hmid); free(acc); free(ct); free(st);
}

/* Prefill of one chunk per sequence after the positions already in the cache.  Sequence b's
 * seq_lens[b] tokens tokens[b][0..len) sit at positions starts[b] .. starts[b] + len - 1 (starts
 * NULL: all 0).  Cache slots 0..starts[b]-1 hold that sequence's earlier keys and values and are
 * read, never written; slots starts[b] .. starts[b]+len-1 are written; the rest stay untouched.
 * Each new position attends every slot up to itself.  last_hidden [B][H] = final RMSNorm of
 * position starts[b] + len_b - 1.  Returns 0, or -1 on a bad argument.
 * Source: batched prefill with KV writes ("Stabilize Higgs Audio termination and prefill",
 * Summary); pads trail and only the used keys are attended (the fp8_chain page, its description);
 * mixed batches of prefill chunks and single-token steps under one launch bound taken from the
 * real batch (vLLM-Omni PR #8226, Purpose). */
static int prefill_impl(const oracle_dims* d, const uint16_t* embed, const oracle_layer* layers,
                        const uint16_t* final_norm, const int32_t* tokens, const int32_t* seq_lens,
                        const int32_t* starts, int B, int P_max, uint16_t* kv, int kv_batch, int n_slots,
                        uint16_t* last_hidden, const oracle_fp8_layer* fp8, float* amax,
                        const oracle_nvfp4_layer* nv4) {
    const int H = d->hidden;
    const size_t blk = (size_t)2 * d->n_kv_heads * n_slots * d->head_dim;
    if (B < 1 || B > kv_batch) return -1;
    for (int b = 0; b < B; ++b) {
        const int n = seq_lens[b], s0 = starts ? starts[b] : 0;
        if (n < 1 || n > P_max || s0 < 0 || s0 + n > n_slots) return -1;
        for (int i = 0; i < n; ++i)
            if (tokens[(size_t)b * P_max + i] < 0 || tokens[(size_t)b * P_max + i] >= d->vocab) return -1;
    }
    for (int b = 0; b < B; ++b) {
        const int n = seq_lens[b], s0 = starts ? starts[b] : 0;
        uint16_t* x = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * H);
        uint16_t* hid = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * H);
        for (int i = 0; i < n; ++i)
            memcpy(x + (size_t)i * H, embed + (size_t)tokens[(size_t)b * P_max + i] * H,
                   sizeof(uint16_t) * H);
        forward_rows(d, layers, final_norm, x, s0, n, kv + (size_t)b * blk, (size_t)kv_batch * blk,
                     n_slots, hid, fp8, amax, nv4);
        memcpy(last_hidden + (size_t)b * H, hid + (size_t)(n - 1) * H, sizeof(uint16_t) * H);
        free(x);
        free(hid);
    }
    return 0;
}

int oracle_prefill_chunk(const oracle_dims* d, const uint16_t* embed, const oracle_layer* layers,
                         const uint16_t* final_norm, const int32_t* tokens, const int32_t* seq_lens,
                         const int32_t* starts, int B, int P_max, uint16_t* kv, int kv_batch, int n_slots,
                         uint16_t* last_hidden) {
    return prefill_impl(d, embed, layers, final_norm, tokens, seq_lens, starts, B, P_max, kv, kv_batch, n_slots,
                        last_hidden, NULL, NULL, NULL);
}

/* FP8 variant of the prefill from position 0: every projection of every layer runs on E4M3 weights
 * fp8[l] and on its input quantized with that layer's static activation scale, the result scaled
 * by activation scale * weight scale; everything else is the bf16 prefill (the fp8_chain page, its
 * description: static-FP8 merged-QKV, output, gate/up and down GEMMs). */
int oracle_prefill_fp8(const oracle_dims* d, const uint16_t* embed, const oracle_layer* layers,
                       const oracle_fp8_layer* fp8, const uint16_t* final_norm, const int32_t* tokens,
                       const int32_t* seq_lens, int B, int P_max, uint16_t* kv, int kv_batch, int n_slots,
                       uint16_t* last_hidden) {
    if (fp8 == NULL) return -1;
    return prefill_impl(d, embed, layers, final_norm, tokens, seq_lens, NULL, B, P_max, kv, kv_batch, n_slots,
                        last_hidden, fp8, NULL, NULL);
}

/* NVFP4-band variant of the prefill from position 0 (the fp8_chain page, its precision bands): the
 * merged QKV in static FP8, the output, gate/up and down projections in NVFP4 -- E2M1 weights with
 * E4M3 block scales and an fp32 global scale, each input quantized per call to E2M1 with block
 * scales from its own data under a static global scale; everything else is the bf16 prefill. */
int oracle_prefill_nvfp4(const oracle_dims* d, const uint16_t* embed, const oracle_layer* layers,
                         const oracle_nvfp4_layer* nv4, const uint16_t* final_norm, const int32_t* tokens,
                         const int32_t* seq_lens, int B, int P_max, uint16_t* kv, int kv_batch, int n_slots,
                         uint16_t* last_hidden) {
    if (nv4 == NULL) return -1;
    if (d->hidden % 16 != 0 || (d->n_q_heads * d->head_dim) % 16 != 0 || d->ffn % 16 != 0) return -1;
    return prefill_impl(d, embed, layers, final_norm, tokens, seq_lens, NULL, B, P_max, kv, kv_batch, n_slots,
                        last_hidden, NULL, NULL, nv4);
}

/* Calibration of the static activation scales (FlashRT PR #141, Summary: FP8 activation scales
 * from a fixed calibration prompt): the bf16 prefill of the calibration batch, recording per layer
 * l the max |x| over every row of each projection's input -- amax[4l + 0..3] for the QKV, output,
 * gate/up and down projections.  The scale of a projection is then amax / 448. */
int oracle_calibrate(const oracle_dims* d, const uint16_t* embed, const oracle_layer* layers,
                     const uint16_t* final_norm, const int32_t* tokens, const int32_t* seq_lens, int B, int P_max,
                     int n_slots, float* amax) {
    for (int i = 0; i < 4 * d->n_layers; ++i) amax[i] = 0.0f;
    const size_t per = (size_t)d->n_layers * B * 2 * d->n_kv_heads * n_slots * d->head_dim;
    uint16_t* kv = (uint16_t*)calloc(per, sizeof(uint16_t));
    uint16_t* last = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)B * d->hidden);
    const int rc = prefill_impl(d, embed, layers, final_norm, tokens, seq_lens, NULL, B, P_max, kv, B, n_slots,
                                last, NULL, amax, NULL);
    free(kv);
    free(last);
    return rc;
}

/* Batched prefill from position 0: tokens [B][P_max] with trailing pads (never read); seq_lens[B]
 * in [1, n_slots].  kv [L][kv_batch][2][nkv][n_slots][hd]: slots 0..len-1 of sequence b are
 * written, others untouched.  last_hidden [B][H] = final RMSNorm of position len_b - 1. */
int oracle_prefill(const oracle_dims* d, const uint16_t* embed, const oracle_layer* layers,
                   const uint16_t* final_norm, const int32_t* tokens, const int32_t* seq_lens,
                   int B, int P_max, uint16_t* kv, int kv_batch, int n_slots, uint16_t* last_hidden) {
    return prefill_impl(d, embed, layers, final_norm, tokens, seq_lens, NULL, B, P_max, kv, kv_batch, n_slots,
                        last_hidden, NULL, NULL, NULL);
}

/* Single-token decode pass: row b is the embedding in_emb[b] at position pos[b]; it writes cache
 * slot pos[b] of every layer and attends slots 0..pos[b].  hidden [B][H] = final RMSNorm output.
 * Source: the AR audio decode pass per frame ("Stabilize Higgs Audio termination and prefill",
 * Performance: AR decode ms/frame); its input is the summed codebook embedding. */
int oracle_decode(const oracle_dims* d, const oracle_layer* layers, const uint16_t* final_norm,
                  const uint16_t* in_emb, const int32_t* pos, int B, uint16_t* kv, int kv_batch,
                  int n_slots, uint16_t* hidden) {
    const int H = d->hidden;
    const size_t blk = (size_t)2 * d->n_kv_heads * n_slots * d->head_dim;
    if (B < 1 || B > kv_batch) return -1;
    for (int b = 0; b < B; ++b)
        if (pos[b] < 0 || pos[b] >= n_slots) return -1;
    for (int b = 0; b < B; ++b)
        forward_rows(d, layers, final_norm, in_emb + (size_t)b * H, pos[b], 1, kv + (size_t)b * blk,
                     (size_t)kv_batch * blk, n_slots, hidden + (size_t)b * H, NULL, NULL, NULL);
    return 0;
}

/* ---------------------------------------------------------------- delayed-codebook step */

/* Delay-pattern state machine for one row, given a chooser for the codebooks that are neither
 * forced to BOS nor to EOC.  state = (frame t, eoc_frame e (-1 none), done, 0), updated in place.
 * Source: per-frame choice with delay handling, and the delayed-EOC fix that makes EOC on any
 * codebook terminate ("Stabilize Higgs Audio termination and prefill", Summary and Root cause).
 * Rule (codebook k lags k frames):
 *   t < k               -> BOS (codebook not started)
 *   e >= 0, t - k >= e  -> EOC (codebook past the end)
 *   otherwise           -> choose(k) (argmax, or a sample)
 *   if e < 0 and some chosen codebook is EOC: e = min over those k of (t - k), and every codebook
 *   with t >= k and t - k >= e is EOC in this frame too
 *   done |= e >= 0 and t >= e + K - 1; t += 1 (a done row keeps advancing and emits all EOC). */
typedef int (*choose_fn)(void* ctx, int b, int k, int t);

static void delay_row(int K, int bos, int eoc, int b, int32_t* st, int32_t* c, int32_t* done, choose_fn choose,
                      void* ctx) {
    int t = st[0], e = st[1], dn = st[2];
    int forced[64];
    for (int k = 0; k < K; ++k) {
        if (t < k) {
            c[k] = bos;
            forced[k] = 1;
        } else if (e >= 0 && t - k >= e) {
            c[k] = eoc;
            forced[k] = 1;
        } else {
            c[k] = choose(ctx, b, k, t);
            forced[k] = 0;
        }
    }
    if (e < 0) {
        int cand = INT_MAX;
        for (int k = 0; k < K; ++k)
            if (!forced[k] && c[k] == eoc && t - k < cand) cand = t - k;
        if (cand != INT_MAX) {
            e = cand;
            for (int k = 0; k < K; ++k)
                if (t >= k && t - k >= e) c[k] = eoc;
        }
    }
    if (e >= 0 && t >= e + K - 1) dn = 1;
    st[0] = t + 1;
    st[1] = e;
    st[2] = dn;
    st[3] = 0;
    *done = dn;
}

typedef struct {
    int K, Vc, eoc;
    const float* logits;
    const float* eoc_bias;
} greedy_ctx;

/* argmax over all Vc logits (eoc_bias[b][k] added to the EOC logit), lowest index on ties */
static int choose_argmax(void* vctx, int b, int k, int t) {
    (void)t;
    const greedy_ctx* g = (const greedy_ctx*)vctx;
    const float* lg = g->logits + ((size_t)b * g->K + k) * g->Vc;
    int best = 0;
    float bv = 0.0f;
    for (int v = 0; v < g->Vc; ++v) {
        float x = lg[v];
        if (v == g->eoc && g->eoc_bias) x = x + g->eoc_bias[(size_t)b * g->K + k];
        if (v == 0 || x > bv) {
            bv = x;
            best = v;
        }
    }
    return best;
}

/* Greedy step for B rows from fp32 logits [B][K][Vc]; codes [B][K]; done [B]; state [B][4]. */
void oracle_delay_step(int K, int Vc, int bos, int eoc, const float* logits, const float* eoc_bias,
                       int B, int32_t* state, int32_t* codes, int32_t* done) {
    greedy_ctx g = {K, Vc, eoc, logits, eoc_bias};
    for (int b = 0; b < B; ++b)
        delay_row(K, bos, eoc, b, state + (size_t)b * 4, codes + (size_t)b * K, done + b, choose_argmax, &g);
}

/* ---------------------------------------------------------------- sampled codebook step */

/* Philox4x32-10 counter-based generator, from its published definition (Salmon, Moraes, Dror,
 * Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011): ten rounds of
 *   (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
 * with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key bumped by the Weyl constants (0x9E3779B9,
 * 0xBB67AE85) between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1, n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Exponential noise of entry v of codebook k at frame t for a row seeded with `seed` (the
 * per-request seeded exponential noise of vLLM-Omni PR #8226, Purpose and Step-overhead
 * reductions): word v & 3 of Philox4x32-10 at counter (v >> 2, k, t, 0) under key
 * (seed low 32 bits, seed high 32 bits), as a uniform u = (x >> 8 + 1) / 2^24 in (0, 1], and
 * E = -log(u) in fp32. */
float oracle_exponential(uint64_t seed, int t, int k, int v) {
    const uint32_t ctr[4] = {(uint32_t)v >> 2, (uint32_t)k, (uint32_t)t, 0u};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    const float u = (float)((out[v & 3] >> 8) + 1u) * (1.0f / 16777216.0f);
    return -logf(u);
}

typedef struct {
    float z;
    int v;
} zv;

/* descending z, then ascending index */
static int cmp_zv(const void* a, const void* b) {
    const zv* x = (const zv*)a;
    const zv* y = (const zv*)b;
    if (x->z > y->z) return -1;
    if (x->z < y->z) return 1;
    return x->v < y->v ? -1 : (x->v > y->v);
}

typedef struct {
    int K, Vc, eoc;
    const float* logits;
    const float* eoc_bias;
    float temperature, top_p;
    int top_k;
    const uint64_t* seeds;
    float* margin;    /* [B][K] or NULL: relative gap of the two fastest race times (-1 if forced) */
    int32_t* amb;     /* [B][K] or NULL: 1 where the top-p cut falls within 1e-4 of an entry's boundary */
} sample_ctx;

/* One sampled code (temperature, top-k, top-p, then the exponential race; vLLM-Omni PR #8226,
 * Purpose and Test Plan: temperature 1, top-k 50, top-p 0.95, seeded exponential noise):
 *   z_v = (logit_v (+ eoc_bias on the EOC entry)) / temperature, fp32;
 *   order the Vc entries by z descending, ties by ascending index;
 *   top-k (0 < top_k < Vc): keep every entry whose z is >= the top_k-th largest z;
 *   top-p (top_p < 1): with p = softmax of z over the kept entries, keep an entry while the
 *     probability of the kept entries before it in that order is < top_p (so the shortest prefix
 *     reaching top_p, and at least the first entry);
 *   exponential race: each kept entry's clock is E_v / q_v with q_v = exp(z_v - z_max) and E_v the
 *     entry's exponential noise; the first clock to ring (smallest, lowest index on ties) is the
 *     sample -- a draw from the kept entries with probability proportional to q_v.
 * Floating point decides the code here, so the oracle takes the decisions in fp32 like the
 * kernel: the comparisons of z are exact, the sums run in the sorted order above. */
static int choose_sample(void* vctx, int b, int k, int t) {
    const sample_ctx* s = (const sample_ctx*)vctx;
    const int Vc = s->Vc;
    const float* lg = s->logits + ((size_t)b * s->K + k) * Vc;
    zv* e = (zv*)malloc(sizeof(zv) * (size_t)Vc);
    for (int v = 0; v < Vc; ++v) {
        float x = lg[v];
        if (v == s->eoc && s->eoc_bias) x = x + s->eoc_bias[(size_t)b * s->K + k];
        const float z = x / s->temperature;
        e[v].z = z != z ? -INFINITY : z;   /* a NaN logit counts as -inf */
        e[v].v = v;
    }
    qsort(e, (size_t)Vc, sizeof(zv), cmp_zv);
    int n = Vc;
    if (s->top_k > 0 && s->top_k < Vc) {
        const float zk = e[s->top_k - 1].z;
        n = s->top_k;
        while (n < Vc && e[n].z >= zk) ++n;
    }
    float* q = (float*)malloc(sizeof(float) * (size_t)n);
    const float zmax = e[0].z;
    float S = 0.0f;
    for (int i = 0; i < n; ++i) {
        q[i] = expf(e[i].z - zmax);
        S += q[i];
    }
    int amb = 0;
    int m = n;
    if (s->top_p < 1.0f) {
        float cum = 0.0f;
        m = 0;
        for (int i = 0; i < n; ++i) {
            if (fabsf(cum - s->top_p) < 1e-4f) amb = 1;
            if (!(cum < s->top_p)) break;
            m = i + 1;
            cum += q[i] / S;
        }
        if (m == 0) m = 1;
    }
    const uint64_t seed = s->seeds[b];
    int best = -1;
    float bt = 0.0f, second = INFINITY;
    for (int i = 0; i < m; ++i) {
        if (q[i] == 0.0f) continue;   /* probability 0 (underflow): its clock never rings */
        const float tv = oracle_exponential(seed, t, k, e[i].v) / q[i];
        if (best < 0 || tv < bt || (tv == bt && e[i].v < best)) {
            if (best >= 0) second = fminf(second, bt);
            bt = tv;
            best = e[i].v;
        } else {
            second = fminf(second, tv);
        }
    }
    if (s->margin) s->margin[(size_t)b * s->K + k] = m > 1 ? (float)(((double)second - bt) / (double)bt) : INFINITY;
    if (s->amb) s->amb[(size_t)b * s->K + k] = amb;
    free(q);
    free(e);
    return best;
}

/* Sampled step for B rows from fp32 logits [B][K][Vc]: the delay state machine with each
 * non-forced codebook sampled by choose_sample with the row's seed seeds[b] and the row's frame t.
 * margin / amb (optional, [B][K]): the near-tie diagnostics of each sampled codebook (margin -1
 * and amb 0 where the slot was forced).  Returns 0, or -1 on a bad argument. */
int oracle_sample_step(int K, int Vc, int bos, int eoc, const float* logits, const float* eoc_bias,
                       float temperature, int top_k, float top_p, const uint64_t* seeds, int B,
                       int32_t* state, int32_t* codes, int32_t* done, float* margin, int32_t* amb) {
    if (B < 1 || K < 1 || K > 64 || Vc < 1 || !(temperature > 0.0f) || !(top_p > 0.0f)) return -1;
    if (margin)
        for (int i = 0; i < B * K; ++i) margin[i] = -1.0f;
    if (amb)
        for (int i = 0; i < B * K; ++i) amb[i] = 0;
    sample_ctx c = {K, Vc, eoc, logits, eoc_bias, temperature, top_p, top_k, seeds, margin, amb};
    for (int b = 0; b < B; ++b)
        delay_row(K, bos, eoc, b, state + (size_t)b * 4, codes + (size_t)b * K, done + b, choose_sample, &c);
    return 0;
}

/* next[b] = bf16(sum over k ascending of fp32 code_emb[k][codes[b][k]]).  code_emb [K][Vc][H].
 * Source: codebook embedding accumulation into the next input ("Stabilize Higgs Audio termination
 * and prefill", Summary). */
void oracle_code_embed_sum(int K, int Vc, int H, const uint16_t* code_emb, const int32_t* codes,
                           int B, uint16_t* next) {
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < H; ++i) {
            float s = 0.0f;
            for (int k = 0; k < K; ++k)
                s += bf(code_emb[((size_t)k * Vc + codes[(size_t)b * K + k]) * H + i]);
            next[(size_t)b * H + i] = to_bf(s);
        }
}

/* Full step: logits[b][k][v] = hidden[b] . head_w[k*Vc + v] (fp32), then the delay state machine,
 * then the embedding sum.  logits_out (optional) receives the raw logits (bias not included). */
int oracle_codebook_step(const oracle_dims* d, const uint16_t* hidden, const uint16_t* head_w,
                         const uint16_t* code_emb, int32_t* state, const float* eoc_bias, int B,
                         int32_t* codes, uint16_t* next, int32_t* done, float* logits_out) {
    const int K = d->n_codebooks, Vc = d->codebook_size, H = d->hidden;
    if (B < 1 || K < 1 || K > 64) return -1;
    float* lg = logits_out ? logits_out : (float*)malloc(sizeof(float) * (size_t)B * K * Vc);
    oracle_linear(hidden, head_w, B, K * Vc, H, lg);
    oracle_delay_step(K, Vc, d->bos_id, d->eoc_id, lg, eoc_bias, B, state, codes, done);
    oracle_code_embed_sum(K, Vc, H, code_emb, codes, B, next);
    if (!logits_out) free(lg);
    return 0;
}

/* Sampled full step: the logits as in oracle_codebook_step, then oracle_sample_step, then the
 * embedding sum of the sampled codes. */
int oracle_codebook_step_sampled(const oracle_dims* d, const uint16_t* hidden, const uint16_t* head_w,
                                 const uint16_t* code_emb, int32_t* state, const float* eoc_bias,
                                 float temperature, int top_k, float top_p, const uint64_t* seeds, int B,
                                 int32_t* codes, uint16_t* next, int32_t* done, float* logits_out) {
    const int K = d->n_codebooks, Vc = d->codebook_size, H = d->hidden;
    if (B < 1 || K < 1 || K > 64) return -1;
    float* lg = logits_out ? logits_out : (float*)malloc(sizeof(float) * (size_t)B * K * Vc);
    oracle_linear(hidden, head_w, B, K * Vc, H, lg);
    const int rc = oracle_sample_step(K, Vc, d->bos_id, d->eoc_id, lg, eoc_bias, temperature, top_k, top_p, seeds,
                                      B, state, codes, done, NULL, NULL);
    if (rc == 0) oracle_code_embed_sum(K, Vc, H, code_emb, codes, B, next);
    if (!logits_out) free(lg);
    return rc;
}
