/*
 * CPU oracle for int8 weight-only Qwen3-family decode -- TEST INFRASTRUCTURE.
 *
 * Only the test suite, the package's smoke check and the benchmark's CPU
 * baseline leg may load this library.  The CUDA library never includes,
 * links or calls it, and it includes nothing from the CUDA library.
 *
 * What it computes: the plain definition of the decoder that the pages name
 * ("Model-agnostic LLM inference", section "Supported models": grouped-query
 * attention with RMSNorm on Q/K, tied embeddings, SiLU-gated FFN, RoPE, no
 * attention bias) over int8 weights with one fp32 scale per output row
 * (same page, section "The quantized load cache"), greedy argmax decode
 * ("Run local LLM decode", section "Limitations": every generated token is
 * the argmax at its step), with a prefill that fills the KV cache from the
 * prompt ("LLM inference overview", section "Results" and "Workload
 * characteristics").  Arithmetic is fp32; the K and V cache entries are
 * rounded to bf16 (round to nearest even) when they are stored, and every
 * attention read (including the entry just stored) uses the rounded value.
 */
#ifndef ORC_H
#define ORC_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t hidden, n_layers, n_heads, n_kv_heads, head_dim, intermediate, vocab;
    float rope_theta, rms_eps;
} orc_dims;

typedef struct {
    const int8_t* q;   /* [out][in] row-major */
    const float* s;    /* [out] */
} orc_mat;

typedef struct {
    orc_mat wq, wk, wv, wo, wg, wu, wd;
    const float *attn_norm, *ffn_norm, *q_norm, *k_norm;
} orc_layer;

typedef struct {
    orc_dims d;
    orc_mat embed;              /* [vocab][hidden], also the lm_head (tied) */
    const orc_layer* layers;    /* [n_layers] */
    const float* final_norm;    /* [hidden] */
} orc_model;

typedef struct orc_cache orc_cache;

/* ---- pieces (each pinned by the oracle's own tests) ---- */
uint16_t orc_bf16_bits(float x);
float orc_bf16_value(uint16_t bits);
void orc_rmsnorm(const float* x, const float* g, int n, float eps, float* y);
void orc_rope(float* v, int hd, int pos, float theta);
float orc_silu(float z);
void orc_matmul_i8(const orc_mat* w, int rows, int cols, const float* x, int m, float* y, int nthreads);
void orc_attention(const float* q, const uint16_t* k, const uint16_t* v, int len, int cap,
                   int n_heads, int n_kv_heads, int hd, float* out);
int orc_argmax(const float* z, int n);

/* ---- whole model ---- */
orc_cache* orc_cache_new(const orc_model* m, int capacity);
void orc_cache_free(orc_cache* c);
int orc_cache_len(const orc_cache* c);
/* copy layer `l` of the cache: [n_kv_heads][len][head_dim] bf16 bits each */
void orc_cache_read(const orc_cache* c, int l, uint16_t* k, uint16_t* v);

/* Run n new tokens at positions len..len+n-1 of the cache (causal), append
 * their K/V, and write logits [(n - logits_from)][vocab] for block rows
 * logits_from..n-1 (logits may be NULL when logits_from >= n).
 * Returns 0, or -1 when the cache would overflow. */
int orc_forward_block(const orc_model* m, orc_cache* c, const int32_t* ids, int n, int logits_from,
                      float* logits, int nthreads);

/* Greedy decode of one sequence: prefill the prompt, then max_new argmax
 * steps (stopping after eos_id when eos_id >= 0).  Returns the count. */
int orc_greedy(const orc_model* m, const int32_t* prompt, int n_prompt, int max_new, int32_t eos_id,
               int32_t* out, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
