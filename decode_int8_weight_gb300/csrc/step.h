// The small-batch decode step (host side of step.cu).
//
// One layer is three kernels chained by programmatic dependent launch:
//   attention block  (clusters of 8 CTAs, one cluster per query head):
//       RMSNorm -> the head's Q rows and its group's K, V rows -> QK-RMSNorm,
//       RoPE, bf16 KV append -> split attention merged inside the cluster ->
//       this head's share of the O projection, added to the residual stream;
//   gate/up          RMSNorm -> gate/up rows -> SiLU(gate) * up;
//   down             down rows, added to the residual stream;
// and the step ends with the lm_head sweep and its argmax.  The residual
// stream is carried between kernels in 64-bit fixed point (value * 2^32),
// so the partial sums of the split projections meet in integer atomic adds
// whose result does not depend on their order.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q3 {

constexpr int kStepMaxBatch = 4;  // sequences per step (one 8-column MMA tile: hi and lo of 4 sequences)
constexpr int kClusterCtas = 8;   // CTAs per query head in the attention block
constexpr int kStepKvChunk = 16;      // K/V positions per shared-memory stage of the attention block

struct AttnBlockArgs {
    int B, H, nh, nkv, cap, kv_stages;
    float eps;
    const uint8_t* wqkv;     // QKV tile blobs, K = H (rows: Wq, then Wk, then Wv)
    const uint8_t* wo;       // O tile blobs, K = nh * hd
    const float* o_scale;    // [H]
    const float* attn_norm;  // [H]
    const float* q_norm;     // [hd]
    const float* k_norm;     // [hd]
    const float2* rope;      // [cap][hd / 2] (cos, sin)
    __nv_bfloat16* kc;       // this layer's K cache [bmax][nkv][cap][hd]
    __nv_bfloat16* vc;       // this layer's V cache
    const int32_t* seq_ids;  // [B] cache slot of each row
    const int32_t* pos;      // [B] position of the new token
    int pos_early;           // positions are final before the wait (not written by the previous kernel)
    const long long* xin;    // [B][H] residual stream in (fixed point), or null: the embedding of tokens
    const int32_t* tokens;   // [B] (layer 0)
    const int8_t* emb;       // [V][H] (layer 0)
    const float* emb_scale;  // [V]
    long long* xa;           // [B][H] residual stream out (fixed point), zero on entry
    int32_t* status;
};

struct FfnGateArgs {
    int B, H, I, tpc;        // tpc: 16-row gate/up tiles per CTA
    float eps;
    const uint8_t* wgu;      // gate/up tile blobs (8 gate rows then the same 8 up units), K = H
    const float* ffn_norm;   // [H]
    const long long* xa;     // [B][H] residual stream (fixed point)
    long long* xf;           // [B][H] next residual accumulator: zeroed here
    __half* ah;              // activation planes (fragment order, 8 column tiles), K = I
    int32_t* status;
};

struct FfnDownArgs {
    int B, H, I, ks;         // ks: K parts per 16-row tile
    const uint8_t* wd;       // down tile blobs, K = I
    const float* d_scale;    // [H]
    const __half* ah;        // activation planes from the gate/up kernel
    long long* xa;           // [B][H] residual in: added by part 0, then zeroed
    long long* xf;           // [B][H] residual out (accumulated)
    int32_t* status;
};

struct LmHeadArgs {
    int B, H, rows, valid_rows, stages;
    float eps;
    const uint8_t* w;        // embedding tile blobs (tied lm_head), K = H
    const float* final_norm; // [H]
    const long long* xf;     // [B][H] residual stream after the last layer
    unsigned long long* keys;// [B] zero between launches
    unsigned int* counter;   // zero between launches
    int32_t* tokens;         // [B] next token
    int32_t* out_ids;        // [B][out_cap]
    int32_t* step;
    int out_cap;
    int32_t* pos;
    int advance_pos;
    float* logits;           // optional [B][valid_rows]
    int32_t* status;
};

struct StepShape {
    int H, I, nh, nkv, hd, vocab_rows;
};

// Shared-memory bytes of each kernel (0 if the shape does not fit).
size_t attn_block_smem(int H, int hd, int kv_stages);
size_t ffn_gate_smem(int H, int tpc);
size_t ffn_down_smem(int I, int ks);
size_t lm_head_smem(int H, int stages);

// Launch geometry chosen for a shape on a device with num_sms SMs.
struct StepPlan {
    int kv_stages = 2;
    int gate_tpc = 1, gate_grid = 1;
    int down_ks = 1, down_grid = 1;
    int lm_stages = 8, lm_grid = 1;
};
bool step_plan(const StepShape& s, int num_sms, int smem_optin, StepPlan* plan);

// Sets the kernels' shared-memory attribute on the current device (once per
// device); false if the device refused.
bool step_prepare_device(const StepShape& s, const StepPlan& p);

cudaError_t launch_attn_block(const AttnBlockArgs& a, int hd, cudaStream_t st);
cudaError_t launch_ffn_gate(const FfnGateArgs& a, int grid, cudaStream_t st);
cudaError_t launch_ffn_down(const FfnDownArgs& a, int grid, cudaStream_t st);
cudaError_t launch_lm_head(const LmHeadArgs& a, int grid, cudaStream_t st);

// Largest number of attention-block clusters of this shape that can be
// resident at once on the current device (0 if none).
int attn_block_max_clusters(int H, int hd, int kv_stages);

}  // namespace q3
