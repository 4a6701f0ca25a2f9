/*
 * CPU oracle for int8 weight-only Qwen3-family decode -- TEST INFRASTRUCTURE.
 * See orc.h for what it computes and who may use it.
 *
 * Plain fp32 C.  Each dot product is summed sequentially in ascending index
 * order; loops over independent outputs may run on several OpenMP threads,
 * which changes no result.  Built with -ffp-contract=off so that no multiply
 * and add are fused and the results do not depend on the host CPU.
 */
#include "orc.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

struct orc_cache {
    orc_dims d;
    int cap, len;
    uint16_t* k; /* [L][n_kv][cap][hd] */
    uint16_t* v;
};

/* ------------------------------------------------------------------ bf16 */

/* Round an fp32 value to the nearest bf16, ties to even (finite inputs). */
uint16_t orc_bf16_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

float orc_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------ RMSNorm
 * "Model-agnostic LLM inference", section "Supported models" (RMSNorm on the
 * hidden state and on Q/K): y = x / sqrt(mean(x^2) + eps) * g. */
void orc_rmsnorm(const float* x, const float* g, int n, float eps, float* y) {
    float ss = 0.0f;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    float inv = 1.0f / sqrtf(ss / (float)n + eps);
    for (int i = 0; i < n; ++i) y[i] = (x[i] * inv) * g[i];
}

/* ------------------------------------------------------------------ RoPE
 * Same section ("RoPE").  Rotate-half pairing (i, i + hd/2), frequency
 * theta^(-2i/hd), angle pos * freq; frequency, angle, cos and sin are taken
 * in double and rounded to fp32, the rotation itself is fp32. */
void orc_rope(float* v, int hd, int pos, float theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double freq = pow((double)theta, -2.0 * (double)i / (double)hd);
        double ang = (double)pos * freq;
        float c = (float)cos(ang), s = (float)sin(ang);
        float a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
    }
}

/* ------------------------------------------------------------------ SiLU
 * Same section ("SiLU-gated FFN"): silu(z) = z / (1 + exp(-z)). */
float orc_silu(float z) { return z / (1.0f + expf(-z)); }

/* ------------------------------------------------------------------ int8 matmul
 * y[t][r] = s[r] * sum_k float(q[r][k]) * x[t][k] for t < m, r < rows,
 * summed over k in ascending order (one accumulator per output).
 * "Model-agnostic LLM inference", section "The quantized load cache": int8
 * weights with one scale per row.  The loop nest keeps, for each output row,
 * up to 64 tokens' accumulators side by side; each accumulator still adds
 * its k terms in order. */
void orc_matmul_i8(const orc_mat* w, int rows, int cols, const float* x, int m, float* y, int nthreads) {
    enum { TB = 64 };
    float* xt = (float*)malloc((size_t)cols * TB * sizeof(float));
    for (int t0 = 0; t0 < m; t0 += TB) {
        int tb = (m - t0 < TB) ? (m - t0) : TB;
        for (int k = 0; k < cols; ++k)
            for (int t = 0; t < tb; ++t) xt[(size_t)k * TB + t] = x[(size_t)(t0 + t) * cols + k];
#pragma omp parallel for schedule(static) num_threads(nthreads)
        for (int r = 0; r < rows; ++r) {
            float acc[TB];
            for (int t = 0; t < tb; ++t) acc[t] = 0.0f;
            const int8_t* qr = w->q + (size_t)r * cols;
            for (int k = 0; k < cols; ++k) {
                float wk = (float)qr[k];
                const float* xk = xt + (size_t)k * TB;
                for (int t = 0; t < tb; ++t) acc[t] += wk * xk[t];
            }
            for (int t = 0; t < tb; ++t) y[(size_t)(t0 + t) * rows + r] = w->s[r] * acc[t];
        }
    }
    free(xt);
}

/* ------------------------------------------------------------------ attention
 * Grouped-query attention for one position: query head j reads kv head
 * j / (n_heads / n_kv_heads); scores q . K[t] / sqrt(hd) over the len cached
 * positions, max-subtracted softmax with expf, output sum_t p_t V[t].
 * k, v: [n_kv][cap][hd] bf16 bits (only the first len positions are read).
 * q: [n_heads][hd]; out: [n_heads][hd]. */
void orc_attention(const float* q, const uint16_t* k, const uint16_t* v, int len, int cap,
                   int n_heads, int n_kv_heads, int hd, float* out) {
    int group = n_heads / n_kv_heads;
    float scale = 1.0f / sqrtf((float)hd);
    float* p = (float*)malloc((size_t)len * sizeof(float));
    for (int j = 0; j < n_heads; ++j) {
        int g = j / group;
        const float* qj = q + (size_t)j * hd;
        const uint16_t* kg = k + (size_t)g * cap * hd;
        const uint16_t* vg = v + (size_t)g * cap * hd;
        float mx = -INFINITY;
        for (int t = 0; t < len; ++t) {
            float dot = 0.0f;
            for (int d = 0; d < hd; ++d) dot += qj[d] * orc_bf16_value(kg[(size_t)t * hd + d]);
            p[t] = dot * scale;
            if (p[t] > mx) mx = p[t];
        }
        float sum = 0.0f;
        for (int t = 0; t < len; ++t) {
            p[t] = expf(p[t] - mx);
            sum += p[t];
        }
        for (int t = 0; t < len; ++t) p[t] = p[t] / sum;
        float* oj = out + (size_t)j * hd;
        for (int d = 0; d < hd; ++d) {
            float acc = 0.0f;
            for (int t = 0; t < len; ++t) acc += p[t] * orc_bf16_value(vg[(size_t)t * hd + d]);
            oj[d] = acc;
        }
    }
    free(p);
}

/* ------------------------------------------------------------------ argmax
 * "Run local LLM decode", section "Limitations": each generated token is the
 * argmax at its step.  Ties go to the lowest index. */
int orc_argmax(const float* z, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (z[i] > z[best]) best = i;
    return best;
}

/* ------------------------------------------------------------------ cache */

orc_cache* orc_cache_new(const orc_model* m, int capacity) {
    orc_cache* c = (orc_cache*)calloc(1, sizeof(orc_cache));
    c->d = m->d;
    c->cap = capacity;
    c->len = 0;
    size_t n = (size_t)m->d.n_layers * m->d.n_kv_heads * capacity * m->d.head_dim;
    c->k = (uint16_t*)calloc(n, sizeof(uint16_t));
    c->v = (uint16_t*)calloc(n, sizeof(uint16_t));
    return c;
}

void orc_cache_free(orc_cache* c) {
    if (!c) return;
    free(c->k);
    free(c->v);
    free(c);
}

int orc_cache_len(const orc_cache* c) { return c->len; }

void orc_cache_read(const orc_cache* c, int l, uint16_t* k, uint16_t* v) {
    int nkv = c->d.n_kv_heads, hd = c->d.head_dim;
    for (int g = 0; g < nkv; ++g)
        for (int t = 0; t < c->len; ++t) {
            size_t src = (((size_t)l * nkv + g) * c->cap + t) * hd;
            size_t dst = ((size_t)g * c->len + t) * hd;
            memcpy(k + dst, c->k + src, (size_t)hd * 2);
            memcpy(v + dst, c->v + src, (size_t)hd * 2);
        }
}

/* ------------------------------------------------------------------ model
 * One decoder pass over n new tokens (prefill when the cache is empty, a
 * decode step when n == 1).  Per layer, in the order the Qwen3 block takes:
 *   h = rmsnorm(x) * g_attn;  q, k, v = Wq h, Wk h, Wv h
 *   per head: q = rmsnorm(q) * g_q, k = rmsnorm(k) * g_k; RoPE at position
 *   store bf16(k), bf16(v); attention over positions 0..pos (causal)
 *   x += Wo o;  h = rmsnorm(x) * g_ffn;  x += Wd (silu(Wg h) * (Wu h))
 * then h = rmsnorm(x) * g_final and logits = E h (tied embedding table). */
int orc_forward_block(const orc_model* m, orc_cache* c, const int32_t* ids, int n, int logits_from,
                      float* logits, int nthreads) {
    const orc_dims d = m->d;
    const int H = d.hidden, I = d.intermediate, hd = d.head_dim;
    const int nh = d.n_heads, nkv = d.n_kv_heads, Dq = nh * hd, Dkv = nkv * hd;
    const int start = c->len;
    if (n <= 0) return 0;
    if (start + n > c->cap) return -1;

    float* x = (float*)malloc((size_t)n * H * sizeof(float));
    float* h = (float*)malloc((size_t)n * H * sizeof(float));
    float* q = (float*)malloc((size_t)n * Dq * sizeof(float));
    float* k = (float*)malloc((size_t)n * Dkv * sizeof(float));
    float* v = (float*)malloc((size_t)n * Dkv * sizeof(float));
    float* o = (float*)malloc((size_t)n * Dq * sizeof(float));
    float* y = (float*)malloc((size_t)n * (H > I ? H : I) * sizeof(float));
    float* gt = (float*)malloc((size_t)n * I * sizeof(float));
    float* up = (float*)malloc((size_t)n * I * sizeof(float));

    /* embedding gather from the tied int8 table */
    for (int t = 0; t < n; ++t) {
        const int8_t* row = m->embed.q + (size_t)ids[t] * H;
        float s = m->embed.s[ids[t]];
        for (int i = 0; i < H; ++i) x[(size_t)t * H + i] = (float)row[i] * s;
    }

    for (int l = 0; l < d.n_layers; ++l) {
        const orc_layer* ly = &m->layers[l];
        for (int t = 0; t < n; ++t) orc_rmsnorm(x + (size_t)t * H, ly->attn_norm, H, d.rms_eps, h + (size_t)t * H);
        orc_matmul_i8(&ly->wq, Dq, H, h, n, q, nthreads);
        orc_matmul_i8(&ly->wk, Dkv, H, h, n, k, nthreads);
        orc_matmul_i8(&ly->wv, Dkv, H, h, n, v, nthreads);

        uint16_t* kc = c->k + (size_t)l * nkv * c->cap * hd;
        uint16_t* vc = c->v + (size_t)l * nkv * c->cap * hd;
        for (int t = 0; t < n; ++t) {
            int pos = start + t;
            float tmp[512];
            for (int j = 0; j < nh; ++j) {
                float* qj = q + (size_t)t * Dq + (size_t)j * hd;
                orc_rmsnorm(qj, ly->q_norm, hd, d.rms_eps, tmp);
                memcpy(qj, tmp, (size_t)hd * sizeof(float));
                orc_rope(qj, hd, pos, d.rope_theta);
            }
            for (int g = 0; g < nkv; ++g) {
                float* kg = k + (size_t)t * Dkv + (size_t)g * hd;
                const float* vg = v + (size_t)t * Dkv + (size_t)g * hd;
                orc_rmsnorm(kg, ly->k_norm, hd, d.rms_eps, tmp);
                memcpy(kg, tmp, (size_t)hd * sizeof(float));
                orc_rope(kg, hd, pos, d.rope_theta);
                for (int e = 0; e < hd; ++e) {
                    kc[((size_t)g * c->cap + pos) * hd + e] = orc_bf16_bits(kg[e]);
                    vc[((size_t)g * c->cap + pos) * hd + e] = orc_bf16_bits(vg[e]);
                }
            }
        }
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
        for (int t = 0; t < n; ++t)
            orc_attention(q + (size_t)t * Dq, kc, vc, start + t + 1, c->cap, nh, nkv, hd, o + (size_t)t * Dq);

        orc_matmul_i8(&ly->wo, H, Dq, o, n, y, nthreads);
        for (size_t i = 0; i < (size_t)n * H; ++i) x[i] = x[i] + y[i];

        for (int t = 0; t < n; ++t) orc_rmsnorm(x + (size_t)t * H, ly->ffn_norm, H, d.rms_eps, h + (size_t)t * H);
        orc_matmul_i8(&ly->wg, I, H, h, n, gt, nthreads);
        orc_matmul_i8(&ly->wu, I, H, h, n, up, nthreads);
        for (size_t i = 0; i < (size_t)n * I; ++i) gt[i] = orc_silu(gt[i]) * up[i];
        orc_matmul_i8(&ly->wd, H, I, gt, n, y, nthreads);
        for (size_t i = 0; i < (size_t)n * H; ++i) x[i] = x[i] + y[i];
    }
    c->len = start + n;

    if (logits && logits_from < n) {
        int nl = n - logits_from;
        for (int t = 0; t < nl; ++t)
            orc_rmsnorm(x + (size_t)(logits_from + t) * H, m->final_norm, H, d.rms_eps, h + (size_t)t * H);
        orc_matmul_i8(&m->embed, d.vocab, H, h, nl, logits, nthreads);
    }
    free(x); free(h); free(q); free(k); free(v); free(o); free(y); free(gt); free(up);
    return 0;
}

int orc_greedy(const orc_model* m, const int32_t* prompt, int n_prompt, int max_new, int32_t eos_id,
               int32_t* out, int nthreads) {
    if (n_prompt <= 0 || max_new <= 0) return 0;
    orc_cache* c = orc_cache_new(m, n_prompt + max_new);
    float* z = (float*)malloc((size_t)m->d.vocab * sizeof(float));
    int count = 0;
    orc_forward_block(m, c, prompt, n_prompt, n_prompt - 1, z, nthreads);
    for (;;) {
        int32_t tok = orc_argmax(z, m->d.vocab);
        out[count++] = tok;
        if (count >= max_new || (eos_id >= 0 && tok == eos_id)) break;
        orc_forward_block(m, c, &tok, 1, 0, z, nthreads);
    }
    free(z);
    orc_cache_free(c);
    return count;
}
