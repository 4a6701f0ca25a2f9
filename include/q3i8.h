/*
 * q3i8 -- int8 weight-only Qwen3-family decode on one NVIDIA GB300 (sm_103a).
 *
 * C ABI of libq3i8.so.  Plain pointers and sizes only.
 *
 * The operation ("Model-agnostic LLM inference" and "Run local LLM decode"):
 * prompt token ids in, greedy generated token ids out, for a Qwen3-family
 * decoder (grouped-query attention with RMSNorm on Q/K, RoPE, SiLU-gated
 * FFN, tied embeddings, no attention bias; "Model-agnostic LLM inference",
 * section "Supported models") whose weights are int8 with one fp32 scale per
 * output row (same page, section "The quantized load cache").  A prefill
 * reads each whole prompt and builds the KV cache; each decode step then
 * sweeps the weights once for all B sequences and ends in an argmax
 * ("LLM inference overview", sections "Results" and "Workload
 * characteristics"; "Run local LLM decode", section "Limitations": greedy,
 * every token is the argmax at its step).  The KV cache is bf16.
 *
 * Numerics: fp32 accumulation over exact int8 weights; K and V are rounded to
 * bf16 (nearest even) when stored and read back rounded.  Argmax ties go to
 * the lowest token id.
 *
 * Errors: every entry point returns a status (Q3_OK == 0).  The message of
 * the last failure on a context is q3i8_last_error(ctx); failures before a
 * context exists put their message in q3i8_last_error(NULL) (per thread).
 * Validation failures are reported before any device work starts.
 *
 * Threading: a context is bound to one device and one CUDA stream and is not
 * thread-safe; use one context per host thread.
 *
 * Groups of calls: the decode context (q3i8_init .. q3i8_destroy); single
 * kernels on caller memory for isolated checks (q3i8_op_*); the quantized
 * load cache (q3i8_cache_*, host only); the continuous-batching scheduler
 * (q3i8_sched_*) and its device loop (q3i8_cb_*, q3i8_sched_run).
 */
#ifndef Q3I8_H
#define Q3I8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
enum {
    Q3_OK = 0,
    /* The model shape is outside the supported family or alignment gates
     * ("Model-agnostic LLM inference", section "Supported models": GQA
     * heads % kv_heads == 0; hidden, intermediate and heads*head_dim each a
     * multiple of 32; tied embeddings; no attention bias).  The message lists
     * every mismatch, not just the first.  These kernels also need
     * head_dim in {64, 128}. */
    Q3_ERR_UNSUPPORTED_ARCH = 1,
    /* Empty or out-of-range prompt ids, max_new_tokens < 1, B outside
     * [1, max_batch], NULL where an array is required ("Model-agnostic LLM
     * inference", section "Errors", invalid_arguments). */
    Q3_ERR_INVALID_ARGUMENTS = 2,
    /* prompt + new tokens above the 65,536-position ceiling ("Model-agnostic
     * LLM inference", section "Long context"). */
    Q3_ERR_CONTEXT = 3,
    /* No CUDA device, or a device that is not sm_103. */
    Q3_ERR_NO_DEVICE = 4,
    /* Device memory allocation failed. */
    Q3_ERR_OOM = 5,
    /* Any other CUDA runtime failure (the message names the call). */
    Q3_ERR_CUDA = 6,
    /* A bounded device-side wait gave up; the kernel returned early and the
     * results of that call are invalid.  The context stays usable. */
    Q3_ERR_TIMEOUT = 7,
    /* Call order: q3i8_step_logits before any prefill, or a step past the
     * context's capacity. */
    Q3_ERR_STATE = 8
};

/* ---------------------------------------------------------------- model */
typedef struct q3i8_dims {
    int32_t hidden;             /* H */
    int32_t n_layers;           /* L */
    int32_t n_heads;            /* query heads */
    int32_t n_kv_heads;         /* key/value heads (GQA) */
    int32_t head_dim;           /* 64 or 128 */
    int32_t intermediate;       /* I (FFN width) */
    int32_t vocab;              /* V (tied embedding rows) */
    float rope_theta;           /* 1e6 for Qwen3 */
    float rms_eps;              /* 1e-6 for Qwen3 */
    int32_t max_batch;          /* most sequences per call, 1..32 */
    int32_t max_ctx;            /* initial per-sequence KV capacity in positions
                                   (0 means 512); raised automatically up to
                                   65,536 when a call needs more */
    int32_t tie_word_embeddings;/* must be 1 */
    int32_t attention_bias;     /* must be 0 */
} q3i8_dims;

/* One linear layer in nn.Linear order: w is [out][in] row-major int8,
 * scale is [out] fp32; y = scale * (w . x). */
typedef struct q3i8_mat {
    const int8_t* w;
    const float* scale;
} q3i8_mat;

/* One decoder layer.  q: [n_heads*head_dim][H], k and v: [n_kv*head_dim][H],
 * o: [H][n_heads*head_dim], gate and up: [I][H], down: [H][I].
 * Norm gains are fp32: attn_norm and ffn_norm [H], q_norm and k_norm
 * [head_dim] (shared by all heads). */
typedef struct q3i8_layer {
    q3i8_mat q, k, v, o, gate, up, down;
    const float* attn_norm;
    const float* ffn_norm;
    const float* q_norm;
    const float* k_norm;
} q3i8_layer;

typedef struct q3i8_stats {
    double prefill_ms;              /* device time of the prefill (CUDA events) */
    double decode_ms;               /* device time of the decode steps */
    double prefill_tokens_per_sec;  /* prompt tokens / prefill time */
    double decode_tokens_per_sec;   /* tokens from decode steps / decode time */
    double step_us;                 /* mean decode step */
    int64_t prefill_tokens;
    int64_t decode_steps;
} q3i8_stats;

typedef struct q3i8_ctx q3i8_ctx;

/* ---------------------------------------------------------------- calls */

/* Host-only check of a model shape against the architecture gates ("Model-
 * agnostic LLM inference", section "Supported models").  Touches no GPU.
 * On failure writes every mismatch, separated by "; ", into msg (always
 * NUL-terminated when msg_cap > 0) and returns Q3_ERR_UNSUPPORTED_ARCH (or
 * Q3_ERR_INVALID_ARGUMENTS for non-positive sizes or a bad max_batch). */
int q3i8_validate_dims(const q3i8_dims* dims, char* msg, size_t msg_cap);

/* Create a context on the current CUDA device.  Copies every weight from
 * the caller's HOST arrays into library-owned device memory (repacked for
 * the kernels), so the caller may free them on return; weights then stay
 * resident for every later call ("Model-agnostic LLM inference", section
 * "Convert once, decode many times": loaded weights stay resident).
 *   embed       [vocab][H] int8 + [vocab] scales: embedding table and, tied,
 *               the lm_head.
 *   layers      [n_layers] host array of layer descriptors.
 *   final_norm  [H] fp32 gain of the last RMSNorm.
 *   cuda_stream cudaStream_t to run on (NULL = a stream the context creates).
 * On success *out receives the context (free with q3i8_destroy). */
int q3i8_init(const q3i8_dims* dims, const q3i8_mat* embed, const q3i8_layer* layers,
              const float* final_norm, void* cuda_stream, q3i8_ctx** out);

/* Greedy decode of B sequences ("Run local LLM decode", section "Read the
 * result"; "LLM inference overview": batched decode sweeps the weights once
 * per step for all B sequences).  HOST buffers:
 *   prompt_ids[b]  pointer to prompt_lens[b] token ids of sequence b.
 *   out_ids        [B][max_new_tokens] generated ids, row b for sequence b.
 *   out_counts     [B] number of valid ids per row: max_new_tokens, or up to
 *                  and including the first eos_id when eos_id >= 0.  With
 *                  eos_id >= 0 decoding stops once every sequence has
 *                  produced it (checked every 16 steps); entries of out_ids
 *                  after a row's count are not meaningful (-1 where no step
 *                  ran).
 *   stats          optional timings (NULL to skip).
 * Resets the KV cache, prefills every prompt, runs max_new_tokens-1 decode
 * steps (each one replay of a captured CUDA graph of the step's kernels) and
 * copies the ids back once at the end.  Context sizing: max(512, longest prompt + new tokens),
 * raised automatically up to 65,536 positions ("Model-agnostic LLM
 * inference", section "Long context"). */
int q3i8_decode(q3i8_ctx* ctx, int32_t B, const int32_t* const* prompt_ids, const int32_t* prompt_lens,
                int32_t max_new_tokens, int32_t eos_id, int32_t* out_ids, int32_t* out_counts,
                q3i8_stats* stats);

/* Settings of the sampling chain ("Model-agnostic LLM inference", section
 * "Sampling": repetition / presence / frequency penalties -> temperature ->
 * top-k -> min-p -> top-p -> a seeded weighted draw).  Readings of the
 * page's names, all in float64 over the model's fp32 logits:
 *   penalties   over the tokens already in the sequence (prompt and earlier
 *               generated tokens), token t seen c times: a positive logit is
 *               divided by repeat_penalty and any other multiplied by it,
 *               then presence_penalty and c * frequency_penalty are
 *               subtracted;
 *   temperature divides the penalised logits; 0 selects the greedy argmax
 *               (every other setting is then ignored);
 *   order       candidates by penalised logit descending, token ascending;
 *   top_k       keeps the first top_k (1 .. 4096);
 *   min_p       keeps candidates whose softmax probability is at least
 *               min_p times the largest ([0, 1], 0 = off);
 *   top_p       keeps the shortest prefix whose softmax probabilities sum
 *               to at least top_p ((0, 1], 1 = off);
 *   draw        u = the top 24 bits of SplitMix64 output c + 1 started at
 *               seed, c = i * 2^20 + b for generated token i of sequence b,
 *               times 2^-24; the token is the first survivor whose
 *               cumulative probability exceeds u.
 * The same settings and seed give the same tokens; top_k = 1 gives the
 * greedy tokens at any temperature. */
typedef struct q3i8_sampling {
    double temperature;
    double top_p;
    double min_p;
    double repeat_penalty;       /* > 0; 1 = off */
    double presence_penalty;
    double frequency_penalty;
    int32_t top_k;
    int32_t reserved;            /* set to 0 */
    uint64_t seed;
} q3i8_sampling;

/* q3i8_decode with every generated token drawn by the sampling chain on the
 * device (the first one included), from `sampling` (HOST struct; NULL is an
 * error; temperature 0 is exactly q3i8_decode).  Each decode step's graph
 * ends with one sampling kernel after the lm_head.  Q3_ERR_INVALID_ARGUMENTS
 * for a setting outside the ranges above or not finite. */
int q3i8_decode_sample(q3i8_ctx* ctx, int32_t B, const int32_t* const* prompt_ids, const int32_t* prompt_lens,
                       int32_t max_new_tokens, int32_t eos_id, const q3i8_sampling* sampling, int32_t* out_ids,
                       int32_t* out_counts, q3i8_stats* stats);

/* As q3i8_decode, with DEVICE buffers: d_prompt_ids holds the B prompts back
 * to back (sum of prompt_lens ids, sequence 0 first); d_out_ids receives
 * [B][max_new_tokens] ids.  prompt_lens stays a host array.  Nothing is
 * copied between host and device except the per-call row tables; returns
 * after the device work has finished. */
int q3i8_decode_device(q3i8_ctx* ctx, int32_t B, const int32_t* d_prompt_ids, const int32_t* prompt_lens,
                       int32_t max_new_tokens, int32_t* d_out_ids, q3i8_stats* stats);

/* Teacher-forced checking interface (the pages' step-by-step session).
 * q3i8_prefill resets the KV cache and runs the B prompts (HOST ids); when
 * last_logits is not NULL it receives the fp32 logits [B][vocab] of each
 * prompt's last position.  Each q3i8_step_logits then appends tokens[b]
 * (HOST, [B]) at the next position of sequence b and writes the fp32 logits
 * [B][vocab] for the position after it into the HOST buffer logits. */
int q3i8_prefill(q3i8_ctx* ctx, int32_t B, const int32_t* const* prompt_ids, const int32_t* prompt_lens,
                 float* last_logits);
int q3i8_step_logits(q3i8_ctx* ctx, const int32_t* tokens, float* logits);

/* Copy the cached K and V (bf16 bit patterns) of one layer and sequence for
 * positions [0, n_pos) into HOST arrays k and v, each [n_kv_heads][n_pos]
 * [head_dim].  For checking. */
int q3i8_read_kv(q3i8_ctx* ctx, int32_t layer, int32_t seq, int32_t n_pos, uint16_t* k, uint16_t* v);

/* Algorithmic HBM bytes of one decode step: weights + scales + norm gains
 * read once, plus the K/V read for sum_b (pos_b + 1) positions and written
 * for B positions. */
int64_t q3i8_step_bytes(const q3i8_ctx* ctx, int32_t B, const int32_t* positions);

/* Kernel launches of one decode step at batch B (the captured graph). */
int32_t q3i8_step_launches(const q3i8_ctx* ctx, int32_t B);

/* Kernels this context has launched so far (graph replays counted per node). */
int64_t q3i8_launch_count(const q3i8_ctx* ctx);

/* Diagnostics: run ONE decode step (as q3i8_step_logits would, without
 * logits) with %globaltimer stamps recorded at every phase boundary of the
 * persistent step kernel, and copy them to the HOST array stamps
 * [grid][stride] (nanoseconds).  *grid and *stride receive the shape.  Needs a
 * prior q3i8_prefill; returns Q3_ERR_STATE when the batch decodes with the
 * chained kernels (the default; the environment variable
 * Q3I8_PERSISTENT_MAX_BATCH=B, read at q3i8_init, selects the persistent
 * kernel up to B sequences) or when cap is too small. */
int q3i8_trace_step(q3i8_ctx* ctx, const int32_t* tokens, uint64_t* stamps, size_t cap, int32_t* grid,
                    int32_t* stride);

const char* q3i8_last_error(const q3i8_ctx* ctx);
const char* q3i8_status_name(int status);
void q3i8_destroy(q3i8_ctx* ctx);

/* ---------------------------------------------------------------- ops
 * Single kernels on caller-owned DEVICE memory, for checking each kernel in
 * isolation.  All run on `cuda_stream` (NULL = legacy default stream) and
 * return after enqueueing (no synchronisation).
 */

/* Dense int8-weight projection on the tcgen05 tensor cores, the contraction
 * of the prefill ("LLM inference overview", section "Workload
 * characteristics": each prompt projection is one wide matmul):
 *   y[m][n] = scale[n] * sum_k w[n][k] * x[m][k],  m < M, n < N.
 *   a_planes [M][2K] f16 bit patterns: row m holds hi(m, 0..K-1) then
 *            lo(m, 0..K-1), with x = hi + lo (hi = f16(x), lo = f16(x - hi)).
 *   w        [N][K] int8 row-major; scale [N] fp32; y [M][N] fp32.
 *   N % 128 == 0, K % 64 == 0, M >= 1; all buffers 16-byte aligned.
 *   d_status device int32 set non-zero if a bounded wait gave up (may be
 *            NULL). */
int q3i8_op_gemm_i8(const uint16_t* a_planes, const int8_t* w, const float* scale, int32_t M, int32_t N, int32_t K,
                    float* y, int32_t* d_status, void* cuda_stream);

/* q3i8_op_gemm_i8 with K split over several CTAs per output tile, as the
 * prefill does when the output tiles alone cannot cover the GPU's SMs (a
 * short prompt on a narrow projection).  Each split writes unscaled fp32
 * partial sums into `workspace`; a second kernel adds them in split order
 * (the result does not depend on which CTA finished first), scales them and
 * stores y.  The split count follows from M, N, K and the current device's
 * SM count; q3i8_op_gemm_i8_splitk_workspace returns the bytes it needs (0
 * when the shape is not split, in which case workspace may be NULL).
 * workspace is 16-byte aligned device memory, no initialisation needed. */
size_t q3i8_op_gemm_i8_splitk_workspace(int32_t M, int32_t N, int32_t K);
int q3i8_op_gemm_i8_splitk(const uint16_t* a_planes, const int8_t* w, const float* scale, int32_t M, int32_t N,
                           int32_t K, float* y, void* workspace, size_t ws_bytes, int32_t* d_status,
                           void* cuda_stream);

/* Split-KV grouped-query decode attention (the attention step of the
 * "Supported models" block, one query position per row):
 *   q       [R][n_heads][hd] fp32 queries (already normed and rotated).
 *   k, v    bf16 caches [n_seq][n_kv][cap][hd] (cap a multiple of 64).
 *   row_seq [R] int32 sequence of each row; row_len [R] int32 positions
 *           0..row_len-1 attended (1 <= row_len <= cap).
 *   out     [R][n_heads][hd] fp32.
 *   splits  KV splits per (row, kv head), 1..64.
 *   workspace, ws_bytes: device scratch for the partial softmax states,
 *           at least q3i8_op_attention_workspace(R, n_heads, hd, splits)
 *           bytes, 16-byte aligned; contents need no initialisation.
 *   d_status device int32 set non-zero if a bounded wait gave up (may be
 *           NULL). */
size_t q3i8_op_attention_workspace(int32_t R, int32_t n_heads, int32_t hd, int32_t splits);
int q3i8_op_attention(const float* q, const uint16_t* k, const uint16_t* v, const int32_t* row_seq,
                      const int32_t* row_len, int32_t R, int32_t n_heads, int32_t n_kv_heads, int32_t hd,
                      int32_t cap, int32_t splits, float* out, void* workspace, size_t ws_bytes,
                      int32_t* d_status, void* cuda_stream);

/* The sampling chain of q3i8_decode_sample on one step's logits:
 *   logits    [B][V] fp32 DEVICE; row b is sequence b.
 *   counts    [B][V] int32 DEVICE: how often each token occurs in sequence b
 *             so far (the penalties' history); the drawn token's count is
 *             incremented.
 *   sampling  HOST settings; temperature must be > 0.
 *   step      the generated-token index i of the draw (u's counter is
 *             i * 2^20 + b).
 *   tokens    [B] int32 DEVICE: receives the drawn tokens.
 *   workspace at least q3i8_op_sample_workspace(B, V) bytes, 16-byte
 *             aligned; no initialisation needed.
 *   d_status  device int32 (may be NULL), set non-zero if the selection is
 *             inconsistent (an internal error).
 * Copies the settings into the workspace and waits for that copy; the draw
 * itself is only enqueued. */
size_t q3i8_op_sample_workspace(int32_t B, int32_t V);
int q3i8_op_sample(const float* logits, int32_t B, int32_t V, int32_t* counts, const q3i8_sampling* sampling,
                   int32_t step, int32_t* tokens, void* workspace, size_t ws_bytes, int32_t* d_status,
                   void* cuda_stream);

/* Upper limit, in bytes, of the scratch q3i8_op_attention_static may use:
 * attention_workspace(R, n_heads, hd, splits) must not exceed it. */
#define Q3I8_OP_ATTENTION_STATIC_SCRATCH_BYTES (4u << 20)

/* q3i8_op_attention without a workspace argument and without allocating.
 * The pages have no counterpart of this call: it exists for callers that
 * cannot hand over device memory, e.g. a plain C host program with no device
 * allocator of its own, or code that must not call cudaMalloc/cudaFree
 * between steps because cudaFree synchronises the whole device.
 *
 * Arguments, layouts and results are those of q3i8_op_attention.  The
 * partial softmax states live in one scratch array compiled into the library
 * (Q3I8_OP_ATTENTION_STATIC_SCRATCH_BYTES per device); nothing in it has to
 * start at zero, since every state is written before it is read.
 *
 * The first call on each device (the caller's current device) looks up the
 * scratch array's device address; make that first call before any stream
 * capture begins.  The address is looked up again when the device's context
 * has changed since (after cudaDeviceReset, for instance), so that call too
 * should come before any capture.  Calls that overlap in time on the same device (two
 * streams, two threads) share the scratch and race: serialise them, e.g. on
 * one stream.  Returns Q3_ERR_INVALID_ARGUMENTS (with a message naming the
 * limit) when the sizes need more scratch than the limit. */
int q3i8_op_attention_static(const float* q, const uint16_t* k, const uint16_t* v, const int32_t* row_seq,
                             const int32_t* row_len, int32_t R, int32_t n_heads, int32_t n_kv_heads, int32_t hd,
                             int32_t cap, int32_t splits, float* out, int32_t* d_status, void* cuda_stream);

/* Check of the device-side time-out path.  The pages have no counterpart of
 * this call; it exists so that the give-up branch of the library's bounded
 * waits can be run on a GPU without faulting or hanging it.
 *
 * Launches one warp that waits on phase 0 of a shared-memory mbarrier
 * through the same bounded wait the attention and prefill kernels use: at
 * most `limit` polls (limit < 0: the kernels' own 2^22; limit 0: give up
 * without polling) and at most about one second of wall time, whichever
 * runs out first.  The phase completes only when `arrive` is non-zero.
 *   d_status     device int32, required; zeroed by the call, then set to
 *                Q3_ERR_TIMEOUT by each thread whose wait gave up.
 *   d_elapsed_ns device uint64 (may be NULL): wall time of thread 0's wait.
 * Synchronises `cuda_stream`.  Returns Q3_OK when the wait saw the phase,
 * Q3_ERR_TIMEOUT when it ran out (the context stays usable), Q3_ERR_CUDA on
 * a launch or copy error. */
int q3i8_op_wait_probe(int32_t arrive, int32_t limit, int32_t* d_status, uint64_t* d_elapsed_ns, void* cuda_stream);

/* ------------------------------------------------------ quantized load cache
 * "Model-agnostic LLM inference", section "The quantized load cache": the
 * post-quantization bytes q3i8_init takes (int8 weights, fp32 per-row scales,
 * fp32 norm gains; about one byte per parameter: 598,230,528 bytes for the
 * Qwen3-0.6B shape) in one file, behind a validity gate of magic + dims +
 * SHA-256 of a caller-chosen manifest (the checkpoint's identity, e.g. its
 * manifest file) + exact length.  A cache that fails the gate is not used:
 * the caller takes its full path and writes a fresh cache.  Decoding from a
 * cache's tables gives byte-identical results, since q3i8_init receives the
 * same bytes.  Payload corruption that keeps the length is not detected (the
 * gate hashes the manifest, not the payload).  Host only; no GPU call. */
typedef struct q3i8_cache q3i8_cache;

/* q3i8_cache_open's gate result */
#define Q3I8_CACHE_VALID 0     /* the cache matches: use it */
#define Q3I8_CACHE_ABSENT 1    /* no readable file at the path */
#define Q3I8_CACHE_BAD_MAGIC 2 /* not a cache file, or another format version */
#define Q3I8_CACHE_DIMS 3      /* written for other dims */
#define Q3I8_CACHE_MANIFEST 4  /* written for another manifest (checkpoint) */
#define Q3I8_CACHE_LENGTH 5    /* truncated or extended */

/* Payload bytes of a cache for these dims (0 for NULL). */
uint64_t q3i8_cache_payload_bytes(const q3i8_dims* dims);

/* Write a cache of the given host arrays (the arguments q3i8_init takes) to
 * `path`: written beside it and renamed into place, so a reader never sees
 * a partial file.  manifest may be NULL when manifest_len is 0.  Returns
 * Q3_ERR_UNSUPPORTED_ARCH for dims the gates of q3i8_validate_dims reject,
 * Q3_ERR_INVALID_ARGUMENTS for a NULL pointer or a failed write. */
int q3i8_cache_write(const char* path, const q3i8_dims* dims, const q3i8_mat* embed, const q3i8_layer* layers,
                     const float* final_norm, const void* manifest, size_t manifest_len);

/* Check the cache at `path` against dims (max_batch and max_ctx are not part
 * of the gate) and the manifest.  *gate receives a Q3I8_CACHE_* code; only
 * for Q3I8_CACHE_VALID is *out set, to a handle owning the file's bytes
 * (free with q3i8_cache_close).  A failed gate returns Q3_OK; errors are
 * NULL arguments (Q3_ERR_INVALID_ARGUMENTS), unsupported dims
 * (Q3_ERR_UNSUPPORTED_ARCH) and host memory (Q3_ERR_OOM). */
int q3i8_cache_open(const char* path, const q3i8_dims* dims, const void* manifest, size_t manifest_len,
                    q3i8_cache** out, int32_t* gate);

/* The cache's arrays as q3i8_init arguments: embed, layers[n_layers] and
 * final_norm point into the handle's memory, valid until q3i8_cache_close. */
int q3i8_cache_tables(const q3i8_cache* cache, q3i8_mat* embed, q3i8_layer* layers, const float** final_norm);

void q3i8_cache_close(q3i8_cache* cache);

/* --------------------------------------------------- continuous batching
 * Host-side scheduler of a continuous batch ("LLM inference overview",
 * section "Workload characteristics": one weight sweep per step serves every
 * sequence in flight; each row of a decode step carries its own sequence
 * slot and position).  Requests wait in a FIFO queue, take the lowest free
 * KV slot between steps, and free it when they finish (max_new_tokens
 * tokens, or eos_id, which is kept).  Host only; no GPU call.
 *
 * One step of the caller's loop:
 *   q3i8_sched_plan            admissions (request, slot) and decode rows
 *                              (request, slot, position, input token);
 *   prefill each admission     into its slot, then
 *   q3i8_sched_complete_prefill with each admission's first token;
 *   decode the rows            then q3i8_sched_complete_step with each
 *                              row's next token, in row order.
 * A sequence occupies prompt_len + max_new_tokens - 1 positions of its slot. */
typedef struct q3i8_sched q3i8_sched;

/* max_batch slots of max_ctx positions each. */
int q3i8_sched_new(int32_t max_batch, int32_t max_ctx, q3i8_sched** out);
void q3i8_sched_destroy(q3i8_sched* sched);

/* Queue a request (the prompt is copied).  Q3_ERR_INVALID_ARGUMENTS for an
 * empty prompt or max_new_tokens < 1, Q3_ERR_CONTEXT when it cannot fit a
 * slot.  *request_id numbers requests from 0 in submission order. */
int q3i8_sched_submit(q3i8_sched* sched, const int32_t* prompt, int32_t prompt_len, int32_t max_new_tokens,
                      int32_t eos_id, int32_t* request_id);

/* Plan the next step.  Arrays hold max_batch entries.  Rows are the
 * sequences in flight in slot order (position = prompt_len + generated - 1,
 * token = the last generated token); admissions are queued requests placed
 * in free slots, which join the rows after their prefill.  Q3_ERR_STATE if
 * the previous plan's prefill or step has not been completed. */
int q3i8_sched_plan(q3i8_sched* sched, int32_t* n_admit, int32_t* admit_request, int32_t* admit_slot,
                    int32_t* n_rows, int32_t* row_request, int32_t* row_slot, int32_t* row_pos,
                    int32_t* row_token);

/* Report the first generated token of admitted requests (any order). */
int q3i8_sched_complete_prefill(q3i8_sched* sched, int32_t n, const int32_t* request_ids,
                                const int32_t* first_tokens);

/* Report the next token of each row of the last plan, in row order. */
int q3i8_sched_complete_step(q3i8_sched* sched, int32_t n_rows, const int32_t* tokens);

/* ---- the same loop on the device.  Slots are the context's KV sequences
 * 0 .. max_batch - 1; the calls below keep every other slot's cache. */

/* Size the KV cache for max_ctx positions per slot (growing it reallocates
 * the cache: every slot's contents are lost, so reserve before serving). */
int q3i8_cb_reserve(q3i8_ctx* ctx, int32_t max_ctx);

/* Prefill n prompts (HOST ids) into the distinct slots[0..n) and write each
 * one's greedy first token to first_tokens[n] (HOST).  Errors: a slot out of
 * range or repeated, an empty or NULL prompt, an id outside the vocabulary
 * (Q3_ERR_INVALID_ARGUMENTS); a prompt longer than the reserved positions
 * (Q3_ERR_CONTEXT); no reserve yet (Q3_ERR_STATE). */
int q3i8_cb_prefill(q3i8_ctx* ctx, int32_t n, const int32_t* slots, const int32_t* const* prompt_ids,
                    const int32_t* prompt_lens, int32_t* first_tokens);

/* One decode step over n rows (HOST arrays): row r appends row_token[r] at
 * position row_pos[r] (>= 1) of slot row_slot[r] (distinct slots), attends
 * positions 0 .. row_pos[r] of that slot and writes the greedy next token to
 * next_tokens[r].  One replay of the step graph at batch n; the rows' slots
 * and positions are device inputs of the graph, so any mix of slots and
 * positions shares it. */
int q3i8_cb_step(q3i8_ctx* ctx, int32_t n, const int32_t* row_slot, const int32_t* row_pos,
                 const int32_t* row_token, int32_t* next_tokens);

/* Drive a scheduler to idle on the device: each round plans, prefills the
 * admissions into their slots, reports their first tokens, runs one step
 * over the plan's rows and reports their next tokens.  Reserves the cache
 * for the scheduler's max_ctx first; its max_batch must not exceed the
 * context's.  stats (optional): host wall time of the prefill and step
 * calls, prompt tokens, steps, and rows per second of decode. */
int q3i8_sched_run(q3i8_ctx* ctx, q3i8_sched* sched, q3i8_stats* stats);

/* 1 when nothing is queued, in flight or awaiting a report. */
int32_t q3i8_sched_idle(const q3i8_sched* sched);

/* A request's generated tokens so far (up to cap written), their count and
 * whether it has finished. */
int q3i8_sched_result(const q3i8_sched* sched, int32_t request_id, int32_t* tokens, int32_t cap, int32_t* n_tokens,
                      int32_t* done);

#ifdef __cplusplus
}
#endif
#endif
