/*
 * CPU oracle for batch-1 greedy decoding of a Llama/Qwen-style dense decoder.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library. The product path (the CUDA
 * library and its binding) never calls it and shares no code with it.
 *
 * What it computes: the plain dense forward pass, one token per step, with
 * greedy selection. The tiled persistent kernel of "Tiles: Scheduling LLM
 * Decoding as a Graph of Tiles" (intro: each operator cut into tiles of output
 * rows, norms and activations folded into neighbouring tiles; nothing decided
 * at run time) is a re-partition of exactly these operations, so the oracle is
 * the unpartitioned definition written out:
 *
 *   x = E[t]
 *   per layer: h = R(rmsnorm(x) * g_attn); q,k,v = W h; [per-head q/k RMSNorm];
 *              RoPE(P); q = R(q); K[P] = R(k); V[P] = R(v);
 *              o_i = R(softmax_t(q_i . K_t / sqrt(d)) . V)  over t = 0..P;
 *              x = R(x + Wo o); h2 = R(rmsnorm(x) * g_ffn);
 *              a = R(silu(Wg h2) * (Wu h2)); x = R(x + Wd a)
 *   hf = R(rmsnorm(x) * g_final); logits = E hf (float, never rounded);
 *   token = argmax (lowest index on ties)
 *
 * R() is float -> bfloat16 round-to-nearest-even. Math is FP32 with BF16
 * weights and BF16 activations at the rounding points above ("History and
 * roadmap", "Where it stands": decode in BFloat16; the Tiles page, "What the
 * code contains": CPU reference with BF16 tolerances). Every dot product is a
 * plain left-to-right sum. OpenMP splits independent output rows and heads
 * across threads; each row is still summed in the same order, so results do
 * not depend on the thread count. Built with -ffp-contract=off.
 *
 * Readings where the pages are silent (RoPE rotate-half pairing, llama3
 * frequency scaling, FP64 angle tables, eps, the attention scale, the GQA head
 * mapping, the causal range 0..P inclusive) are stated at each function.
 *
 * Parity pins: whole-model logits have no printed reference values ("parity
 * unpinned" beyond the closed forms and invariants checked in the tests).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, max_pos;
    int qk_norm;       /* per-head RMSNorm on q and k before RoPE (Qwen3 shapes) */
    int rope_scaling;  /* 0 none, 1 llama3 frequency scaling */
    double rope_theta, rs_factor, rs_low, rs_high, rs_orig_max;
    float rms_eps;
} orc_model;

typedef struct {
    const uint16_t *attn_norm, *wq, *wk, *wv, *q_norm, *k_norm, *wo, *ffn_norm, *w_gate,
        *w_up, *w_down;
} orc_layer;

/* Weight-only INT8 copies of one layer's matrices (codes [rows][cols] and one
 * FP32 scale per output row), made by orc_quantize_rows. */
typedef struct {
    const int8_t *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
    const float *sq, *sk, *sv, *so, *s_gate, *s_up, *s_down;
} orc_qlayer;

/* ------------------------------------------------------------------ bf16 */

/* float -> bfloat16 bits, round to nearest, ties to even; NaN stays NaN. */
uint16_t orc_bf16_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16, lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

float orc_f32_from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* round a float vector to bf16 values, in place (kept as float) */
static void round_vec(float *v, int n) {
    for (int i = 0; i < n; ++i) v[i] = orc_f32_from_bf16(orc_bf16_from_f32(v[i]));
}

void orc_bf16_round_array(const float *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_f32(in[i]);
}

/* ------------------------------------------------------------------ RMSNorm */

/* out[i] = (x[i] * r) * g[i], r = 1 / sqrt(sum(x^2) / n + eps), all FP32,
 * the sum taken left to right. Not rounded here; callers round with R(). */
void orc_rmsnorm(const float *x, const uint16_t *g, int n, float eps, float *out) {
    float ss = 0.0f;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    float mean = ss / (float)n;
    float r = 1.0f / sqrtf(mean + eps);
    for (int i = 0; i < n; ++i) out[i] = (x[i] * r) * orc_f32_from_bf16(g[i]);
}

/* ------------------------------------------------------------------ RoPE */

/* Inverse frequencies omega_j = theta^(-2j/d), j < d/2, in FP64; with llama3
 * scaling (reading: the published rule, wavelength lambda = 2 pi / omega):
 *   lambda < orig/high        -> omega
 *   lambda > orig/low         -> omega / factor
 *   otherwise, s = (orig/lambda - low) / (high - low):
 *                                (1 - s) omega / factor + s omega          */
void orc_rope_inv_freq(const orc_model *m, double *inv_freq) {
    int d = m->head_dim;
    for (int j = 0; j < d / 2; ++j) {
        double w = 1.0 / pow(m->rope_theta, (2.0 * j) / (double)d);
        if (m->rope_scaling == 1) {
            double lam = 2.0 * M_PI / w;
            double hi_wl = m->rs_orig_max / m->rs_high;
            double lo_wl = m->rs_orig_max / m->rs_low;
            if (lam < hi_wl) {
                /* high frequency: unchanged */
            } else if (lam > lo_wl) {
                w = w / m->rs_factor;
            } else {
                double s = (m->rs_orig_max / lam - m->rs_low) / (m->rs_high - m->rs_low);
                w = (1.0 - s) * w / m->rs_factor + s * w;
            }
        }
        inv_freq[j] = w;
    }
}

/* cos/sin of angle pos * omega_j, angle and trig in FP64, stored as FP32. */
void orc_rope_cos_sin(const orc_model *m, int pos, float *cos_out, float *sin_out) {
    int h = m->head_dim / 2;
    double *w = (double *)malloc(sizeof(double) * h);
    orc_rope_inv_freq(m, w);
    for (int j = 0; j < h; ++j) {
        double a = (double)pos * w[j];
        cos_out[j] = (float)cos(a);
        sin_out[j] = (float)sin(a);
    }
    free(w);
}

/* Rotate-half pairing (reading: element j pairs with j + d/2, as in the
 * Hugging Face layout the pages load without transposes):
 *   v'[j]       = v[j] cos_j - v[j + d/2] sin_j
 *   v'[j + d/2] = v[j + d/2] cos_j + v[j] sin_j                              */
void orc_rope_apply(float *v, int d, const float *c, const float *s) {
    int h = d / 2;
    for (int j = 0; j < h; ++j) {
        float a = v[j], b = v[j + h];
        v[j] = a * c[j] - b * s[j];
        v[j + h] = b * c[j] + a * s[j];
    }
}

/* ------------------------------------------------------------------ GEMV */

/* y[r] = sum_j W[r][j] x[j], W bf16 row-major [rows][cols], sum left to right.
 *
 * Built with -DORC_ALT_SUM_ORDER, the same sum is taken in another order
 * (eight interleaved partial sums, then added pairwise). That build is not a
 * second definition: it measures how far an equally valid FP32 summation order
 * moves the whole decoder (the floating-point noise floor the GPU path is held
 * to on deep models), nothing else. */
void orc_gemv(const uint16_t *W, int rows, int cols, const float *x, float *y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint16_t *w = W + (int64_t)r * cols;
#ifdef ORC_ALT_SUM_ORDER
        float pa[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j = 0; j < cols; ++j) pa[j & 7] += orc_f32_from_bf16(w[j]) * x[j];
        y[r] = ((pa[0] + pa[1]) + (pa[2] + pa[3])) + ((pa[4] + pa[5]) + (pa[6] + pa[7]));
#else
        float acc = 0.0f;
        for (int j = 0; j < cols; ++j) acc += orc_f32_from_bf16(w[j]) * x[j];
        y[r] = acc;
#endif
    }
}

/* ------------------------------------------------------------------ INT8 weights */

/* Weight-only INT8 with one FP32 scale per output row ("History and roadmap",
 * "Milestones": weight-only INT8 linear layers; the pages give no scheme, so
 * the plainest one): scale_r = max_j |W_rj| / 127, q_rj = round(W_rj / scale_r)
 * to nearest, ties to even, clamped to [-127, 127]; an all-zero row gets scale
 * 0 and codes 0. Everything in FP32 (W is BF16, exact in FP32). */
void orc_quantize_rows(const uint16_t *W, int rows, int cols, int8_t *Q, float *scale) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint16_t *w = W + (int64_t)r * cols;
        float amax = 0.0f;
        for (int j = 0; j < cols; ++j) {
            const float a = fabsf(orc_f32_from_bf16(w[j]));
            if (a > amax) amax = a;
        }
        const float s = amax / 127.0f;
        scale[r] = s;
        for (int j = 0; j < cols; ++j) {
            float qf = s > 0.0f ? rintf(orc_f32_from_bf16(w[j]) / s) : 0.0f;
            if (qf > 127.0f) qf = 127.0f;
            if (qf < -127.0f) qf = -127.0f;
            Q[(int64_t)r * cols + j] = (int8_t)qf;
        }
    }
}

/* y[r] = scale[r] * sum_j Q[r][j] x[j]: the products are exact in FP32 (an
 * 8-bit code times a BF16 value), summed left to right (or, in the
 * ORC_ALT_SUM_ORDER build, in eight interleaved partial sums), then scaled. */
void orc_gemv_q8(const int8_t *Q, const float *scale, int rows, int cols, const float *x, float *y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const int8_t *q = Q + (int64_t)r * cols;
#ifdef ORC_ALT_SUM_ORDER
        float pa[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j = 0; j < cols; ++j) pa[j & 7] += (float)q[j] * x[j];
        const float acc = ((pa[0] + pa[1]) + (pa[2] + pa[3])) + ((pa[4] + pa[5]) + (pa[6] + pa[7]));
#else
        float acc = 0.0f;
        for (int j = 0; j < cols; ++j) acc += (float)q[j] * x[j];
#endif
        y[r] = scale[r] * acc;
    }
}

/* ------------------------------------------------------------------ attention */

/* One query head over positions 0..n-1 of one KV head ([n][d] bf16 rows):
 *   s_t = (q . K_t) * scale; p = softmax(s) (max-subtracted, FP32);
 *   out = sum_t p_t V_t.  Not rounded here.                                 */
void orc_attention(const float *q, const uint16_t *K, const uint16_t *V, int n, int d,
                   float scale, float *out) {
    float *s = (float *)malloc(sizeof(float) * (n > 0 ? n : 1));
    float mx = -INFINITY;
    for (int t = 0; t < n; ++t) {
        const uint16_t *k = K + (int64_t)t * d;
        float dot = 0.0f;
        for (int j = 0; j < d; ++j) dot += q[j] * orc_f32_from_bf16(k[j]);
        s[t] = dot * scale;
        if (s[t] > mx) mx = s[t];
    }
    float l = 0.0f;
    for (int t = 0; t < n; ++t) {
        s[t] = expf(s[t] - mx);
        l += s[t];
    }
    for (int j = 0; j < d; ++j) out[j] = 0.0f;
    for (int t = 0; t < n; ++t) {
        float p = s[t] / l;
        const uint16_t *v = V + (int64_t)t * d;
        for (int j = 0; j < d; ++j) out[j] += p * orc_f32_from_bf16(v[j]);
    }
    free(s);
}

/* ------------------------------------------------------------------ INT8 KV cache */

/* INT8 KV cache with smoothed keys ("History and roadmap": the M8 log's INT8
 * KV cache with smoothed keys, and "Tried and not kept": INT8 tensor cores for
 * Q K^T were dropped because quantizing the queries undid what key smoothing
 * gained, so queries stay unquantized). The pages give no scheme; the plainest
 * one is taken:
 *   - mu[h][j], the key shift of KV head h: the mean over the prefilled
 *     positions 0..n-1 of the BF16 keys of channel j (FP32; 0 when n = 0);
 *   - every cached row x (a key minus mu, or a value) gets one FP32 scale
 *     s = max_j |x_j| / 127 and codes c_j = x_j / s rounded to nearest, ties
 *     to even, clamped to [-127, 127] (an all-zero row: s = 0, codes 0);
 *   - attention reads K_t = s_t c_t and V_t likewise. The shift is not added
 *     back: it adds q . mu to every score of a query, and a softmax does not
 *     change when every score moves by the same amount.                    */
void orc_kv8_quantize_row(const float *x, int d, int8_t *c, float *s_out) {
    float amax = 0.0f;
    for (int j = 0; j < d; ++j) {
        const float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    const float s = amax / 127.0f;
    *s_out = s;
    for (int j = 0; j < d; ++j) {
        float qf = s > 0.0f ? rintf(x[j] / s) : 0.0f;
        if (qf > 127.0f) qf = 127.0f;
        if (qf < -127.0f) qf = -127.0f;
        c[j] = (int8_t)qf;
    }
}

/* mu[j] = (sum_t K[t][j]) / n over n bf16 rows of d (FP64 sum, FP32 result). */
void orc_kv8_key_mean(const uint16_t *K, int n, int d, float *mu) {
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int t = 0; t < n; ++t) acc += (double)orc_f32_from_bf16(K[(int64_t)t * d + j]);
        mu[j] = n > 0 ? (float)(acc / n) : 0.0f;
    }
}

/* The INT8 form of a [L][n_kv][max_pos][d] cache pair: codes kq, vq (same
 * shape), scales ks, vs ([L][n_kv][max_pos]) and key shifts mu ([L][n_kv][d]). */
typedef struct {
    int8_t *kq, *vq;
    float *ks, *vs, *mu;
} orc_kv8;

/* Fills kv8 from the BF16 caches for positions 0..n_pos-1 (the prefill):
 * mu from those keys, then every row quantized as above. */
void orc_kv8_from_bf16(const orc_model *m, const uint16_t *k_cache, const uint16_t *v_cache, int n_pos,
                       orc_kv8 *kv8) {
    const int d = m->head_dim, heads = m->n_layers * m->n_kv_heads;
    float *row = (float *)malloc(sizeof(float) * d);
    for (int hh = 0; hh < heads; ++hh) {
        const int64_t base = (int64_t)hh * m->max_pos;
        float *mu = kv8->mu + (int64_t)hh * d;
        orc_kv8_key_mean(k_cache + base * d, n_pos, d, mu);
        for (int t = 0; t < n_pos; ++t) {
            const int64_t r = base + t;
            for (int j = 0; j < d; ++j) row[j] = orc_f32_from_bf16(k_cache[r * d + j]) - mu[j];
            orc_kv8_quantize_row(row, d, kv8->kq + r * d, kv8->ks + r);
            for (int j = 0; j < d; ++j) row[j] = orc_f32_from_bf16(v_cache[r * d + j]);
            orc_kv8_quantize_row(row, d, kv8->vq + r * d, kv8->vs + r);
        }
    }
    free(row);
}

/* orc_attention over the INT8 rows: s_t = (q . (ks_t Kq_t)) * scale, then the
 * same softmax and sum_t p_t (vs_t Vq_t). Dequantized values are formed in
 * FP32 (a code times a scale, one rounding), the sums left to right. */
void orc_attention_kv8(const float *q, const int8_t *Kq, const float *Ks, const int8_t *Vq,
                       const float *Vs, int n, int d, float scale, float *out) {
    float *s = (float *)malloc(sizeof(float) * (n > 0 ? n : 1));
    float mx = -INFINITY;
    for (int t = 0; t < n; ++t) {
        const int8_t *k = Kq + (int64_t)t * d;
        float dot = 0.0f;
        for (int j = 0; j < d; ++j) dot += q[j] * (Ks[t] * (float)k[j]);
        s[t] = dot * scale;
        if (s[t] > mx) mx = s[t];
    }
    float l = 0.0f;
    for (int t = 0; t < n; ++t) {
        s[t] = expf(s[t] - mx);
        l += s[t];
    }
    for (int j = 0; j < d; ++j) out[j] = 0.0f;
    for (int t = 0; t < n; ++t) {
        const float p = s[t] / l;
        const int8_t *v = Vq + (int64_t)t * d;
        for (int j = 0; j < d; ++j) out[j] += p * (Vs[t] * (float)v[j]);
    }
    free(s);
}

/* Split-KV form of the same quantity (test helper, used to pin the reading that
 * split partials plus a separate combine equal the unsplit softmax; "History
 * and roadmap", M5 split-KV decode kernels and "Tried and not kept": separate
 * combine). Positions are cut into n_split contiguous ranges [b_c, b_{c+1});
 * per range: m_c = max s, l_c = sum e^{s - m_c}, o_c = sum e^{s - m_c} V;
 * combine: M = max m_c, out = sum e^{m_c - M} o_c / sum e^{m_c - M} l_c.   */
void orc_attention_split(const float *q, const uint16_t *K, const uint16_t *V, int n, int d,
                         float scale, int n_split, const int *bounds, float *out) {
    (void)n; /* bounds[n_split] == n */
    float *m = (float *)malloc(sizeof(float) * n_split);
    float *l = (float *)malloc(sizeof(float) * n_split);
    float *o = (float *)calloc((size_t)n_split * d, sizeof(float));
    for (int c = 0; c < n_split; ++c) {
        int b0 = bounds[c], b1 = bounds[c + 1];
        float mx = -INFINITY;
        for (int t = b0; t < b1; ++t) {
            float dot = 0.0f;
            for (int j = 0; j < d; ++j) dot += q[j] * orc_f32_from_bf16(K[(int64_t)t * d + j]);
            float st = dot * scale;
            if (st > mx) mx = st;
        }
        float lc = 0.0f;
        for (int t = b0; t < b1; ++t) {
            float dot = 0.0f;
            for (int j = 0; j < d; ++j) dot += q[j] * orc_f32_from_bf16(K[(int64_t)t * d + j]);
            float e = expf(dot * scale - mx);
            lc += e;
            for (int j = 0; j < d; ++j) o[(int64_t)c * d + j] += e * orc_f32_from_bf16(V[(int64_t)t * d + j]);
        }
        m[c] = mx;
        l[c] = lc;
    }
    float M = -INFINITY;
    for (int c = 0; c < n_split; ++c)
        if (m[c] > M) M = m[c];
    float L = 0.0f;
    for (int j = 0; j < d; ++j) out[j] = 0.0f;
    for (int c = 0; c < n_split; ++c) {
        if (bounds[c + 1] <= bounds[c]) continue;
        float w = expf(m[c] - M);
        L += w * l[c];
        for (int j = 0; j < d; ++j) out[j] += w * o[(int64_t)c * d + j];
    }
    for (int j = 0; j < d; ++j) out[j] /= L;
    free(m);
    free(l);
    free(o);
}

/* ------------------------------------------------------------------ decoder */

static float silu(float z) { return z / (1.0f + expf(-z)); }

/*
 * Runs n_prompt - 1 + n_new steps. Step s runs at position start_pos + s; its
 * input is prompt[s] for s < n_prompt, otherwise the token chosen at step s-1
 * (or force_tokens[s - n_prompt] when force_tokens is given: teacher forcing,
 * a diagnostic). Steps s >= n_prompt - 1 write out_tokens[s - n_prompt + 1].
 * Caches are [L][n_kv][max_pos][d] bf16, read at positions 0..P and written
 * at P. out_logits ([steps][vocab]) and out_gap ([steps], top-1 minus top-2
 * logit) may be NULL. With qlayers (and lm_q, lm_s for the tied LM head) the
 * GEMVs use those INT8 weights (orc_gemv_q8); the embedding lookup stays BF16.
 * With kv8 (filled for the prefill by orc_kv8_from_bf16), every new K/V row is
 * also quantized into it and attention reads the INT8 cache (orc_attention_kv8);
 * the BF16 caches are still written. Returns 0, or -1 on bad arguments.
 */
int orc_decode(const orc_model *m, const orc_layer *layers, const uint16_t *embed,
               const uint16_t *final_norm, uint16_t *k_cache, uint16_t *v_cache,
               const int32_t *prompt, int n_prompt, int start_pos, int n_new,
               const int32_t *force_tokens, int32_t *out_tokens, float *out_logits,
               float *out_gap, int n_threads, const orc_qlayer *qlayers,
               const int8_t *lm_q, const float *lm_s, orc_kv8 *kv8) {
    if (!m || !layers || !embed || !final_norm || !k_cache || !v_cache || !prompt ||
        n_prompt < 1 || n_new < 0 || start_pos < 0)
        return -1;
    const int steps = n_prompt - 1 + n_new;
    if (start_pos + steps > m->max_pos) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    const int H = m->hidden, F = m->ffn, d = m->head_dim, nq = m->n_q_heads,
              nkv = m->n_kv_heads, V = m->vocab, L = m->n_layers;
    const int G = nq / nkv, qd = nq * d, kvd = nkv * d;
    const float scale = (float)(1.0 / sqrt((double)d));

    float *x = malloc(sizeof(float) * H), *h = malloc(sizeof(float) * H);
    float *q = malloc(sizeof(float) * qd), *k = malloc(sizeof(float) * kvd),
          *v = malloc(sizeof(float) * kvd), *o = malloc(sizeof(float) * qd);
    float *y = malloc(sizeof(float) * (H > F ? H : F));
    float *g = malloc(sizeof(float) * F), *u = malloc(sizeof(float) * F),
          *a = malloc(sizeof(float) * F);
    float *cs = malloc(sizeof(float) * d / 2), *sn = malloc(sizeof(float) * d / 2);
    float *logits = malloc(sizeof(float) * V);
    float *tmp = malloc(sizeof(float) * d);

    int32_t tok = prompt[0];
    int rc = 0;
    for (int s = 0; s < steps; ++s) {
        const int P = start_pos + s;
        if (s < n_prompt) tok = prompt[s];
        else if (force_tokens) tok = force_tokens[s - n_prompt];
        if (tok < 0 || tok >= V) {
            rc = -1;
            break;
        }

        for (int i = 0; i < H; ++i) x[i] = orc_f32_from_bf16(embed[(int64_t)tok * H + i]);
        orc_rope_cos_sin(m, P, cs, sn);

        for (int l = 0; l < L; ++l) {
            const orc_layer *w = &layers[l];
            uint16_t *Kl = k_cache + (int64_t)l * nkv * m->max_pos * d;
            uint16_t *Vl = v_cache + (int64_t)l * nkv * m->max_pos * d;

            orc_rmsnorm(x, w->attn_norm, H, m->rms_eps, h);
            round_vec(h, H);
            const orc_qlayer *qw = qlayers ? &qlayers[l] : NULL;
            if (qw) {
                orc_gemv_q8(qw->wq, qw->sq, qd, H, h, q);
                orc_gemv_q8(qw->wk, qw->sk, kvd, H, h, k);
                orc_gemv_q8(qw->wv, qw->sv, kvd, H, h, v);
            } else {
                orc_gemv(w->wq, qd, H, h, q);
                orc_gemv(w->wk, kvd, H, h, k);
                orc_gemv(w->wv, kvd, H, h, v);
            }
            for (int i = 0; i < nq; ++i) {
                if (m->qk_norm) {
                    orc_rmsnorm(q + i * d, w->q_norm, d, m->rms_eps, tmp);
                    memcpy(q + i * d, tmp, sizeof(float) * d);
                }
                orc_rope_apply(q + i * d, d, cs, sn);
            }
            for (int i = 0; i < nkv; ++i) {
                if (m->qk_norm) {
                    orc_rmsnorm(k + i * d, w->k_norm, d, m->rms_eps, tmp);
                    memcpy(k + i * d, tmp, sizeof(float) * d);
                }
                orc_rope_apply(k + i * d, d, cs, sn);
            }
            round_vec(q, qd);
            for (int i = 0; i < nkv; ++i)
                for (int j = 0; j < d; ++j) {
                    int64_t off = ((int64_t)i * m->max_pos + P) * d + j;
                    Kl[off] = orc_bf16_from_f32(k[i * d + j]);
                    Vl[off] = orc_bf16_from_f32(v[i * d + j]);
                }
            if (kv8) {
                /* the new row, as cached (R(k) - mu, R(v)), into the INT8 cache */
                for (int i = 0; i < nkv; ++i) {
                    const int64_t r = ((int64_t)l * nkv + i) * m->max_pos + P;  /* row in kv8 */
                    const int64_t off = ((int64_t)i * m->max_pos + P) * d;      /* row in Kl, Vl */
                    const float *mu = kv8->mu + ((int64_t)l * nkv + i) * d;
                    for (int j = 0; j < d; ++j) tmp[j] = orc_f32_from_bf16(Kl[off + j]) - mu[j];
                    orc_kv8_quantize_row(tmp, d, kv8->kq + r * d, kv8->ks + r);
                    for (int j = 0; j < d; ++j) tmp[j] = orc_f32_from_bf16(Vl[off + j]);
                    orc_kv8_quantize_row(tmp, d, kv8->vq + r * d, kv8->vs + r);
                }
            }
            /* q head i reads KV head floor(i / G); positions 0..P inclusive */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < nq; ++i) {
                int gi = i / G;
                if (kv8) {
                    const int64_t r0 = ((int64_t)l * nkv + gi) * m->max_pos;
                    orc_attention_kv8(q + i * d, kv8->kq + r0 * d, kv8->ks + r0, kv8->vq + r0 * d,
                                      kv8->vs + r0, P + 1, d, scale, o + i * d);
                } else {
                    orc_attention(q + i * d, Kl + (int64_t)gi * m->max_pos * d,
                                  Vl + (int64_t)gi * m->max_pos * d, P + 1, d, scale, o + i * d);
                }
            }
            round_vec(o, qd);
            if (qw) orc_gemv_q8(qw->wo, qw->so, H, qd, o, y);
            else orc_gemv(w->wo, H, qd, o, y);
            for (int i = 0; i < H; ++i) x[i] = orc_f32_from_bf16(orc_bf16_from_f32(x[i] + y[i]));

            orc_rmsnorm(x, w->ffn_norm, H, m->rms_eps, h);
            round_vec(h, H);
            if (qw) {
                orc_gemv_q8(qw->w_gate, qw->s_gate, F, H, h, g);
                orc_gemv_q8(qw->w_up, qw->s_up, F, H, h, u);
            } else {
                orc_gemv(w->w_gate, F, H, h, g);
                orc_gemv(w->w_up, F, H, h, u);
            }
            for (int i = 0; i < F; ++i) a[i] = silu(g[i]) * u[i];
            round_vec(a, F);
            if (qw) orc_gemv_q8(qw->w_down, qw->s_down, H, F, a, y);
            else orc_gemv(w->w_down, H, F, a, y);
            for (int i = 0; i < H; ++i) x[i] = orc_f32_from_bf16(orc_bf16_from_f32(x[i] + y[i]));
        }

        orc_rmsnorm(x, final_norm, H, m->rms_eps, h);
        round_vec(h, H);
        if (lm_q) orc_gemv_q8(lm_q, lm_s, V, H, h, logits);
        else orc_gemv(embed, V, H, h, logits);
        int best = 0;
        for (int r = 1; r < V; ++r)
            if (logits[r] > logits[best]) best = r;
        if (out_gap) {
            float second = -INFINITY;
            for (int r = 0; r < V; ++r)
                if (r != best && logits[r] > second) second = logits[r];
            out_gap[s] = logits[best] - second;
        }
        if (out_logits) memcpy(out_logits + (int64_t)s * V, logits, sizeof(float) * V);
        if (s >= n_prompt - 1) out_tokens[s - (n_prompt - 1)] = best;
        tok = best;
    }
    free(x); free(h); free(q); free(k); free(v); free(o); free(y);
    free(g); free(u); free(a); free(cs); free(sn); free(logits); free(tmp);
    return rc;
}
