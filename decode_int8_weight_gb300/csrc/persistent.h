// Parameters of the persistent decode-step kernel (host and device).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q3i8.h"

namespace q3 {

// 8-byte word {payload (low 32 bits), epoch flag (high 32 bits)} written with
// one 64-bit store, so a reader that sees the flag also sees the payload.
struct LLw {
    unsigned long long raw;
};

struct PParams {
    int B, bmax, H, I, L, nh, nkv, hd, cap, vocab, vpad, qkv_rows, ns, kmax;
    float eps;
    const uint8_t* const* mats;   // [L*4] tile blobs: qkv, o, gate/up, down
    const uint8_t* lm;            // tile blobs of the tied embedding (lm_head)
    const int8_t* emb_raw;        // [vocab][H] for the embedding gather
    const float* emb_scale;       // [vocab]
    const float* const* gains;    // [L*4]: attn, ffn, q, k
    const float* final_norm;
    const float2* rope;           // [cap][hd/2] (cos, sin)
    __nv_bfloat16* kc;            // [L][bmax][nkv][cap][hd]
    __nv_bfloat16* vc;
    int32_t* tokens;              // [bmax] token of this step -> next token
    int32_t* pos;                 // [bmax] position of this step's token
    int32_t* step;                // output column of this step
    int32_t* out_ids;             // [bmax][out_cap]
    int out_cap;
    int advance_pos;
    uint32_t* epoch;              // step epoch of the flagged words (starts at 1)
    unsigned long long* keys;     // [bmax] argmax keys, zero between steps
    unsigned int* exit_cnt;       // CTAs done with the lm_head, zero between steps
    unsigned int* attn_cnt;       // [L][bmax][nkv] splits done, zero between steps
    int32_t* status;              // 0, or 7 when a bounded wait gave up
    int32_t* abort_flag;          // raised with status; ends every wait in the grid
    int32_t* diag;                // [8] first failed wait: site, cta, warp, layer, phase, aux
    unsigned long long* trace;    // optional [grid][trace_stride] globaltimer stamps
    float* logits;                // optional [B][vocab]
    LLw* x;                       // [bmax][H] residual stream
    LLw* pl_attn;                 // [bmax][H] {hi, lo} of g * x feeding QKV / lm_head
    LLw* pl_ffn;                  // [bmax][H] {hi, lo} of g_ffn * x feeding gate/up
    LLw* ss_attn;                 // [H/16][bmax] per-tile sums of x^2
    LLw* ss_ffn;                  // [H/16][bmax]
    LLw* qkv;                     // [bmax][qkv_rows] fp32 projections
    LLw* pl_o;                    // [bmax][nh*hd] {hi, lo} of the attention output
    LLw* pl_a;                    // [bmax][I] {hi, lo} of silu(gate) * up
    float* part;                  // [bmax][nkv][grid+1][2][hd+2] split-KV softmax states
};

// Trace record of one CTA: [0] start, [1] embedding done, per layer l at
// 2 + 6l: QKV, attention, O, gate/up, down done and the producer's last
// issue of the layer; then the lm_head done and the exit; then up to 32
// (time, event) pairs inside layer kTraceDetailLayer (event = 16 * phase +
// {1: input staged, 2: tile GEMV done, 3: tile epilogue done}).
constexpr int kTraceDetailLayer = 5;
__host__ __device__ inline int trace_detail_base(int L) { return 4 + 6 * L; }
__host__ __device__ inline int trace_stride(int L) { return 4 + 6 * L + 64; }

bool persistent_supported(const q3i8_dims& d);
int persistent_slots(int max_optin_smem, int B, int kmax);
cudaError_t launch_persistent_step(const PParams& P, int grid, cudaStream_t st);

}  // namespace q3
