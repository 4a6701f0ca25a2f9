// Internal state of a q3i8 context (host side of libq3i8.so).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <map>
#include <string>
#include <vector>

#include "../../include/q3i8.h"
#include "step.h"
#include "sample.h"

namespace q3 {
constexpr int kMaxBatch = 32;      // GEMV activation operand: 4 sequences per 8-column MMA tile, 8 tiles
constexpr int kCtxCeiling = 65536; // "Model-agnostic LLM inference", section "Long context"
constexpr int kChunkPos = 64;      // KV positions per attention stage; the cache capacity is a multiple

struct DevMat {
    int8_t* raw = nullptr;     // [rows][cols] row-major int8 (embedding gather, prefill tensor-core GEMM)
    uint8_t* frag = nullptr;   // fragment-order bytes (decode GEMV)
    float* scale = nullptr;    // [rows]
    int rows = 0, valid_rows = 0, cols = 0;
};

struct DevLayer {
    DevMat qkv, o, gu, down;   // qkv: Wq;Wk;Wv rows.  gu: 16-row blocks of 8 gate + 8 up units
    float *attn_norm = nullptr, *ffn_norm = nullptr, *q_norm = nullptr, *k_norm = nullptr;
};
}  // namespace q3

struct q3i8_ctx {
    q3i8_dims d{};
    int dev = 0, num_sms = 0, bmax = 0;
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    std::string err;
    size_t weight_bytes_dev = 0;

    q3::DevMat embed;
    std::vector<q3::DevLayer> layers;
    float* final_norm = nullptr;

    // KV cache [L][bmax][n_kv][cap][hd] bf16 and the RoPE table [cap][hd/2]
    int cap = 0, cap_request = 512;
    __nv_bfloat16 *kc = nullptr, *vc = nullptr;
    float2* rope = nullptr;

    // per-step device state
    int32_t *tokens = nullptr, *pos = nullptr, *seq_ids = nullptr, *step = nullptr, *status = nullptr;
    unsigned long long* keys = nullptr;
    unsigned int* counter = nullptr;
    float* kpart = nullptr;            // split-K parts of the residual GEMVs
    long long* ss_fold = nullptr;      // [2][bmax] folded RMSNorm sums of squares (fixed point)
    unsigned int* tile_cnt = nullptr;  // their per-tile arrival counters
    int attn_resident = 0;             // decode attention CTAs resident at once on the device
    int32_t* out_ids = nullptr;  // [bmax][out_cap]
    int out_cap = 0;

    // decode activations
    float *x = nullptr, *qkv = nullptr, *part = nullptr, *logits = nullptr;
    __half *xh = nullptr, *oh = nullptr, *ah = nullptr;
    int dec_splits_max = 64;

    // prefill buffers (grow-only)
    int pf_rows = 0;
    float *pf_x = nullptr, *pf_qkv = nullptr, *pf_q = nullptr, *pf_part = nullptr;
    __half *pf_xh = nullptr, *pf_oh = nullptr, *pf_ah = nullptr;  // [2M][K] hi/lo planes of the prompt rows
    int4* pf_blocks = nullptr;  // query blocks of the tensor-core prefill attention
    int pf_blocks_cap = 0;
    int32_t *pf_ids = nullptr, *pf_seq = nullptr, *pf_pos = nullptr, *pf_last = nullptr;
    float* pf_work = nullptr;  // split-K partial sums of the prefill projections
    size_t pf_work_bytes = 0;

    // persistent decode step (one cooperative kernel per step)
    bool use_persistent = false;
    int p_max_batch = 0;  // largest B decoded by the persistent kernel; larger B take the chained kernels
    int p_grid = 0, p_ns = 0, p_kmax = 0, p_optin = 0;
    const uint8_t** d_mats = nullptr;     // device [L*4]
    const float** d_gains = nullptr;      // device [L*4]
    uint32_t* p_epoch = nullptr;
    unsigned long long* p_keys = nullptr;
    unsigned int *p_exit = nullptr, *p_attn_cnt = nullptr;
    int32_t* p_abort = nullptr;
    int32_t* p_diag = nullptr;
    unsigned long long* p_trace = nullptr;  // set only for a traced step
    void* p_ll = nullptr;                 // all flagged-word buffers
    float* p_part = nullptr;
    size_t p_ll_bytes = 0;

    // small-batch decode step (step.cu): two cluster kernels per layer
    bool use_step = false;
    int step_max_batch = 0;  // largest B decoded by it; larger B take the chained kernels
    int step_max_ctx = 0;    // longest context (positions) it serves; longer calls take the chained kernels
    int call_ctx = 0;        // longest context the current call can reach
    q3::StepPlan splan;
    long long *xa = nullptr, *xf = nullptr;  // residual stream accumulators [2][bmax][H], value * 2^32

    // seeded sampling (sample.cu), allocated by the first sampling call
    bool seq_ids_custom = false;           // continuous-batching steps pointed the decode rows at other slots
    bool sampling = false;                 // the running call samples instead of taking the argmax
    q3::SampleParams* s_params = nullptr;  // device copy of the call's settings
    int32_t* s_counts = nullptr;           // [bmax][vocab] occurrences of each token per sequence
    uint64_t* s_band_key = nullptr;        // [bmax][sample_band_entries(vocab)] selection scratch
    int32_t* s_band_tok = nullptr;

    std::map<int, cudaGraphExec_t> graphs;  // decode step graph per batch size
    cudaEvent_t ev0 = nullptr, ev1 = nullptr, ev2 = nullptr;

    int64_t launches = 0;        // kernels launched (graph replays counted per node)
    int active_B = 0;            // sequences of the last prefill
    std::vector<int> seq_len;    // host copy of each sequence's filled positions
};

int upload_matrix(q3i8_ctx* c, const std::vector<const int8_t*>& row_src, const std::vector<float>& scales, int K,
                  int pad_rows, q3::DevMat* m, bool keep_raw);
int init_weights(q3i8_ctx* c, const q3i8_mat* embed, const q3i8_layer* layers, const float* final_norm);
int init_state(q3i8_ctx* c);
int ensure_capacity(q3i8_ctx* c, int need_ctx);
void drop_graphs(q3i8_ctx* c);
int decode_splits(const q3i8_ctx* c, int B);
int enqueue_step(q3i8_ctx* c, int B, bool want_logits);
int step_setup(q3i8_ctx* c);
int enqueue_step_fused(q3i8_ctx* c, int B, bool want_logits);
void enqueue_lm_head(q3i8_ctx* c, int B, bool advance_pos, float* logits, const long long* ss_in = nullptr);
int step_launches(const q3i8_ctx* c, int B);
int persistent_setup(q3i8_ctx* c);
int persistent_reset(q3i8_ctx* c);
cudaError_t enqueue_persistent(q3i8_ctx* c, int B, float* logits, unsigned long long* trace = nullptr);
constexpr int kResidSplit = 4;    // K parts per tile of the decode step's residual GEMVs (O, down)
constexpr int kPrefillChunk = 32;  // prompt rows per weight sweep of a prefill projection on the GEMV
// prefills longer than this many rows run their projections on the tcgen05 GEMM
int prefill_launches(const q3i8_ctx* c, int M);
