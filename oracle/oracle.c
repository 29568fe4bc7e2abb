/*
 * Oracle for the DiT attention core -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU definitions of what the GPU path computes.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load this
 * library; the product path never does.  It shares no code, header or table
 * with the CUDA sources.
 *
 * Every tensor is a contiguous fp64 array.  Layouts:
 *   activations  [B, S, H, D]      (BSHD, as the DiT produces them before the
 *                                   pages' transpose to BNSD)
 *   rotary table [S, D/2]          one (cos, sin) per interleaved pair
 *   LSE          [B, H, Sq]
 *   partials     [C, B, Sq, H, D] and [C, B, H, Sq]
 *
 * Sources (page title, section):
 *   RMSNorm  -- "Cosmos Ascend NPU multi-card parallel optimisation notes",
 *               section 3.2 (RMSNorm operator optimisation): y = x * rsqrt(mean(x^2) + eps) * weight;
 *               "NPU Wan2.2-I2V model inference optimisation practice",
 *               section "NPU rms_norm operator adaptation" (WanRMSNorm).
 *   RoPE     -- same Wan2.2 page, section "NPU rotary_mul operator adaptation":
 *               rotary_mode="interleave" with precomputed cos/sin; Cosmos
 *               page section 3.3 (apply_rotary_pos_emb via cos/sin of freqs).
 *   Attention-- same Wan2.2 page, section "NPU npu_fused_infer_attention_score
 *               operator adaptation": non-causal multi-head softmax(scale*QK^T)V
 *               whose second output is the log-sum-exp.  Causal masking (query
 *               i sees keys j <= i) is the VLM attention of the Cosmos page,
 *               section 3.1 (npu_fusion_attention with sparse_mode=2 /
 *               scaled_dot_product_attention with is_causal=True), and the
 *               Wan2.2 page's next_tokens=0 for the causal case.
 *   LSE merge-- "feat: support Ascend NPU backend (torch_npu) for Qwen-Image
 *               pipelines - #274", item 2 (models/basic/attention.py: the ring
 *               path combines per-block outputs with update_out_and_lse); the
 *               Wan2.2 page section "Ring Attention Overlap" (two attention
 *               outputs combined by log-sum-exp).
 *
 * Every function is pinned by the `-m "not gpu"` tests (closed forms,
 * invariants, library routines); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Per-row RMSNorm over the last dimension D: y_d = x_d * w_d / sqrt(mean_d x_d^2 + eps). */
void oracle_rms_norm(const double *x, const double *w, int64_t rows, int64_t D, double eps, double *y) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * D;
        double *yr = y + r * D;
        double ss = 0.0;
        for (int64_t d = 0; d < D; ++d) ss += xr[d] * xr[d];
        double ms = ss / (double)D;
        double inv = 1.0 / sqrt(ms + eps);
        for (int64_t d = 0; d < D; ++d) yr[d] = xr[d] * inv * w[d];
    }
}

/*
 * LayerNorm with adaLN modulation over the last dimension C of x [B, L, C]:
 *   mu = mean_c x_c,  var = mean_c (x_c - mu)^2        (biased variance)
 *   y_c = (x_c - mu) / sqrt(var + eps) * (1 + scale[b, c]) + shift[b, c]
 * scale / shift are [B, C] (one modulation per sample); either may be NULL (0).
 * "NPU Wan2.2-I2V model inference optimisation practice", section
 * "NPU layer_norm_eval operator adaptation" (WanLayerNorm without affine
 * parameters, and FusedLayerNormModulate passing 1 + scale as the weight and
 * shift as the bias of one layer-norm call).
 */
void oracle_layer_norm_modulate(const double *x, const double *scale, const double *shift,
                                int64_t B, int64_t L, int64_t C, double eps, double *y) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < B * L; ++r) {
        const int64_t b = r / L;
        const double *xr = x + r * C;
        double *yr = y + r * C;
        double sum = 0.0;
        for (int64_t c = 0; c < C; ++c) sum += xr[c];
        const double mu = sum / (double)C;
        double ss = 0.0;
        for (int64_t c = 0; c < C; ++c) ss += (xr[c] - mu) * (xr[c] - mu);
        const double inv = 1.0 / sqrt(ss / (double)C + eps);
        for (int64_t c = 0; c < C; ++c) {
            const double sc = scale ? scale[b * C + c] : 0.0, sh = shift ? shift[b * C + c] : 0.0;
            yr[c] = (xr[c] - mu) * inv * (1.0 + sc) + sh;
        }
    }
}

/*
 * Interleaved rotary embedding of x [B, S, H, D]: the pair (x_{2i}, x_{2i+1})
 * at sequence position s is rotated by the angle whose cosine and sine are
 * cos_tab[s, i], sin_tab[s, i]:
 *   y_{2i}   = x_{2i} c - x_{2i+1} s
 *   y_{2i+1} = x_{2i} s + x_{2i+1} c
 */
void oracle_rope_interleaved(const double *x, const double *cos_tab, const double *sin_tab,
                             int64_t B, int64_t S, int64_t H, int64_t D, double *y) {
    const int64_t P = D / 2;
    #pragma omp parallel for schedule(static)
    for (int64_t bs = 0; bs < B * S; ++bs) {
        int64_t s = bs % S;
        for (int64_t h = 0; h < H; ++h) {
            const double *xr = x + (bs * H + h) * D;
            double *yr = y + (bs * H + h) * D;
            for (int64_t i = 0; i < P; ++i) {
                double c = cos_tab[s * P + i], sn = sin_tab[s * P + i];
                double a = xr[2 * i], b = xr[2 * i + 1];
                yr[2 * i] = a * c - b * sn;
                yr[2 * i + 1] = a * sn + b * c;
            }
        }
    }
}

/* The prologue as the pages chain it: RMSNorm over each head's D channels, then interleaved RoPE. */
void oracle_qk_norm_rope(const double *x, const double *w, const double *cos_tab, const double *sin_tab,
                         int64_t B, int64_t S, int64_t H, int64_t D, double eps, double *y) {
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(B * S * H * D));
    if (!tmp) return;
    oracle_rms_norm(x, w, B * S * H, D, eps, tmp);
    oracle_rope_interleaved(tmp, cos_tab, sin_tab, B, S, H, D, y);
    free(tmp);
}

/*
 * Attention of query rows `rows[0..nrows)` (all Sq rows when rows == NULL)
 * over the keys j in [kv_begin, kv_end) -- with `causal`, only keys j <= i
 * (query index i; top-left aligned, as an is_causal scaled-dot-product
 * attention masks):
 *   s_j  = scale * sum_d q_d k_{j,d}
 *   m    = max_j s_j,  l = sum_j exp(s_j - m)
 *   o    = sum_j exp(s_j - m) v_j / l
 *   lse  = m + ln l                    (natural log, scale included)
 * A row with no visible key gives o = 0 and lse = -inf.
 * Outputs: o [B, nrows, H, D], lse [B, H, nrows].
 */
void oracle_attention_masked(const double *q, const double *k, const double *v,
                             int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t D,
                             double scale, int64_t kv_begin, int64_t kv_end, int causal,
                             const int64_t *rows, int64_t nrows, double *o, double *lse) {
    if (rows == NULL) nrows = Sq;
    const int64_t n = kv_end - kv_begin;
    const int64_t total = B * H * nrows;
    #pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t t = 0; t < total; ++t) {
            int64_t r = t % nrows, h = (t / nrows) % H, b = t / (nrows * H);
            int64_t qi = rows ? rows[r] : r;
            const double *qr = q + ((b * Sq + qi) * H + h) * D;
            double *orow = o + ((b * nrows + r) * H + h) * D;
            for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
            if (n <= 0) {
                lse[(b * H + h) * nrows + r] = -INFINITY;
                continue;
            }
            /* keys visible to this row: all of the range, or (causal) those at index <= qi */
            int64_t nv = n;
            if (causal) nv = qi - kv_begin + 1 < n ? qi - kv_begin + 1 : n;
            if (nv <= 0) {
                lse[(b * H + h) * nrows + r] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int64_t j = 0; j < nv; ++j) {
                const double *kr = k + ((b * Skv + kv_begin + j) * H + h) * D;
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d) dot += qr[d] * kr[d];
                sc[j] = scale * dot;
                if (sc[j] > m) m = sc[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nv; ++j) {
                double p = exp(sc[j] - m);
                const double *vr = v + ((b * Skv + kv_begin + j) * H + h) * D;
                for (int64_t d = 0; d < D; ++d) orow[d] += p * vr[d];
                l += p;
            }
            for (int64_t d = 0; d < D; ++d) orow[d] /= l;
            lse[(b * H + h) * nrows + r] = m + log(l);
        }
        free(sc);
    }
}

void oracle_attention(const double *q, const double *k, const double *v,
                      int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t D,
                      double scale, int64_t kv_begin, int64_t kv_end,
                      const int64_t *rows, int64_t nrows, double *o, double *lse) {
    oracle_attention_masked(q, k, v, B, H, Sq, Skv, D, scale, kv_begin, kv_end, 0, rows, nrows, o, lse);
}

/* Softmax probabilities P[b, h, i, j] = exp(s_ij - m_i) / l_i over keys [kv_begin, kv_end) (tiny shapes only). */
void oracle_attention_probs(const double *q, const double *k,
                            int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t D,
                            double scale, int64_t kv_begin, int64_t kv_end, double *p) {
    const int64_t n = kv_end - kv_begin;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < Sq; ++i) {
                const double *qr = q + ((b * Sq + i) * H + h) * D;
                double *pr = p + ((b * H + h) * Sq + i) * n;
                double m = -INFINITY;
                for (int64_t j = 0; j < n; ++j) {
                    const double *kr = k + ((b * Skv + kv_begin + j) * H + h) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d) dot += qr[d] * kr[d];
                    pr[j] = scale * dot;
                    if (pr[j] > m) m = pr[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j < n; ++j) { pr[j] = exp(pr[j] - m); l += pr[j]; }
                for (int64_t j = 0; j < n; ++j) pr[j] /= l;
            }
}

/*
 * Blockwise LSE merge of C partial results (O_c, L_c), each the attention of
 * the same queries over a disjoint key block:
 *   L = m' + ln sum_c exp(L_c - m'),  m' = max_c L_c
 *   O = sum_c exp(L_c - L) O_c
 * Blocks with L_c = -inf carry no weight; if every L_c = -inf then O = 0 and
 * L = -inf.
 * Inputs o_parts [C, B, Sq, H, D], lse_parts [C, B, H, Sq]; outputs o [B, Sq, H, D], lse [B, H, Sq].
 */
void oracle_merge_lse(const double *o_parts, const double *lse_parts,
                      int64_t C, int64_t B, int64_t H, int64_t Sq, int64_t D,
                      double *o, double *lse) {
    const int64_t part_o = B * Sq * H * D, part_l = B * H * Sq;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < B * H * Sq; ++t) {
        int64_t qi = t % Sq, h = (t / Sq) % H, b = t / (Sq * H);
        int64_t li = (b * H + h) * Sq + qi;
        int64_t oi = ((b * Sq + qi) * H + h) * D;
        double mx = -INFINITY;
        for (int64_t c = 0; c < C; ++c)
            if (lse_parts[c * part_l + li] > mx) mx = lse_parts[c * part_l + li];
        for (int64_t d = 0; d < D; ++d) o[oi + d] = 0.0;
        if (mx == -INFINITY) {
            lse[li] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int64_t c = 0; c < C; ++c) sum += exp(lse_parts[c * part_l + li] - mx);
        double L = mx + log(sum);
        for (int64_t c = 0; c < C; ++c) {
            double wgt = exp(lse_parts[c * part_l + li] - L);
            for (int64_t d = 0; d < D; ++d) o[oi + d] += wgt * o_parts[c * part_o + oi + d];
        }
        lse[li] = L;
    }
}

/*
 * ---------------------------------------------------------------- W8A8 fp8
 * "feat: support Ascend NPU backend (torch_npu) for Qwen-Image pipelines -
 * #274", item 4 (npu_quant_linear): activations are quantised per token
 * (dynamic, one scale per row), weights per output channel, to fp8 e4m3; the
 * quantised matmul multiplies the integer-like codes and applies the per-token
 * and per-channel scales, producing bf16.
 *
 * e4m3 (OCP 8-bit floating point, "E4M3"): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9; no
 * infinities; S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448.
 */
double oracle_e4m3_decode(int code) {
    const int sgn = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Round x to the nearest e4m3 value (ties to the even code), saturating to +-448. */
int oracle_e4m3_encode(double x) {
    int sgn = x < 0 || (x == 0 && signbit(x));
    double a = fabs(x);
    if (a >= 448.0) return (sgn << 7) | 0x7E;
    /* walk the 127 non-negative finite codes: they are ordered by value */
    int best = 0;
    double best_err = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_decode(c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (sgn << 7) | best;
}

/*
 * Per-token dynamic quantisation of x [M, K]: scale_m = max_k |x_mk| / 448
 * (1 when the row is all zero), code_mk = e4m3(x_mk / scale_m).  The quotient
 * x / scale decides the code, so it is formed as the kernel forms it: both
 * the scale and the quotient rounded to fp32.
 */
void oracle_quant_fp8_rows(const double *x, int64_t M, int64_t K, unsigned char *codes, float *scale) {
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = (float)fabs(x[m * K + k]);
            if (a > amax) amax = a;
        }
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[m] = sc;
        for (int64_t k = 0; k < K; ++k) {
            float qv = (float)x[m * K + k] / sc;
            codes[m * K + k] = (unsigned char)oracle_e4m3_encode((double)qv);
        }
    }
}

/* out[m, n] = a_scale[m] * b_scale[n] * sum_k dec(a[m, k]) * dec(b[n, k])  (a [M, K], b [N, K] codes) */
void oracle_gemm_fp8(const unsigned char *a, const float *a_scale, const unsigned char *b, const float *b_scale,
                     int64_t M, int64_t N, int64_t K, double *out) {
    double lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = oracle_e4m3_decode(c);
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += lut[a[m * K + k]] * lut[b[n * K + k]];
            out[m * N + n] = acc * (double)a_scale[m] * (double)b_scale[n];
        }
}

