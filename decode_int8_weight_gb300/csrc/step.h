// The small-batch decode step (host side of step.cu).
//
// One layer is two kernels chained by programmatic dependent launch:
//   attention block  (one cluster of 8 CTAs per query head):
//       RMSNorm -> the head's Q rows and its group's K, V rows -> QK-RMSNorm,
//       RoPE, bf16 KV append -> split attention merged inside the cluster ->
//       this head's share of the O projection, added to the residual stream;
//   FFN block        (one CTA per 32 FFN units, no cluster):
//       RMSNorm -> the units' gate/up rows (K whole) -> SiLU(gate) * up ->
//       the units' k-pair of every down row, added to the residual stream;
// and the step ends with the lm_head sweep and its argmax.  Inside an
// attention cluster the 8 CTAs split K of the cluster's rows; their partial
// sums (and the RMSNorm's partial sums of squares) meet in distributed
// shared memory.  The residual stream is carried between kernels in 64-bit
// fixed point (value * 2^32), so the CTAs' shares meet in integer atomic
// adds whose result does not depend on their order.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q3 {

constexpr int kStepMaxBatch = 4;  // sequences per step (one 8-column MMA tile: hi and lo of 4 sequences)
constexpr int kClusterCtas = 8;   // CTAs per cluster
constexpr int kStepKvChunk = 16;  // K/V positions per shared-memory stage of the attention block
constexpr int kFfnUnits = 32;     // FFN units per CTA of the FFN block (4 gate/up tiles; one k-pair of each down row)
constexpr int kFfnResidRows = 64; // most residual rows an FFN CTA adds the stream's input to

struct AttnBlockArgs {
    int B, H, nh, nkv, cap, kv_stages, vocab;
    float eps;
    const uint8_t* wqkv;     // QKV tile blobs, K = H (rows: Wq, then Wk, then Wv)
    const float* qkv_scale;  // [nh hd + 2 nkv hd]
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
    const int32_t* tokens;   // [B] (first layer)
    const int8_t* emb;       // [V][H] (first layer)
    const float* emb_scale;  // [V]
    long long* xa;           // [B][H] residual stream out (fixed point), zero on entry
    long long* clear0;       // [B][H] accumulators this kernel clears for later kernels (may be null)
    long long* clear1;
    int32_t* status;
};

struct FfnBlockArgs {
    int B, H, I;
    float eps;
    const uint8_t* wgu;      // gate/up tile blobs (8 gate rows then the same 8 up units), K = H
    const float* gu_scale;   // [2 I] in tile order
    const uint8_t* wd;       // down tile blobs, K = I
    const float* d_scale;    // [H]
    const float* ffn_norm;   // [H]
    const long long* xa;     // [B][H] residual stream in (fixed point)
    long long* xf;           // [B][H] residual stream out, zero on entry
    int32_t* status;
};

struct LmHeadArgs {
    int B, H, rows, valid_rows, stages;
    float eps;
    const uint8_t* w;        // embedding tile blobs (tied lm_head), K = H
    const float* final_norm; // [H]
    const long long* xf;     // [B][H] residual stream after the last layer
    long long* clear;        // [B][H] accumulator this kernel clears for the next step (may be null)
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

// Shared-memory bytes of each kernel.
size_t attn_block_smem(int H, int hd, int kv_stages);
size_t ffn_block_smem(int H);
size_t lm_head_smem(int H, int stages);

// Launch geometry chosen for a shape on a device.
struct StepPlan {
    int kv_stages = 2;
    int ffn_grid = 1;
    int lm_stages = 6, lm_grid = 1;  // lm_stages <= 8 (one consumer warp per stage)
};
bool step_plan(const StepShape& s, int num_sms, int smem_optin, StepPlan* plan);

// Sets the kernels' shared-memory attribute on the current device (once per
// device); false if the device refused.
bool step_prepare_device();

cudaError_t launch_attn_block(const AttnBlockArgs& a, int hd, cudaStream_t st);
cudaError_t launch_ffn_block(const FfnBlockArgs& a, int grid, cudaStream_t st);
cudaError_t launch_lm_head(const LmHeadArgs& a, int grid, cudaStream_t st);

// Largest number of clusters of each kernel that can be resident at once on
// the current device (0 if none).
int attn_block_max_clusters(int H, int hd, int kv_stages);
int ffn_block_max_blocks(int H);  // FFN blocks resident per SM (0: cannot launch)

}  // namespace q3
