// Launchers of the q3i8 kernels (host side, internal to libq3i8.so).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q3 {

// Packed int8 weight layout of the decode GEMVs ("tile blobs"): one blob per
// 16-row tile, 128 + 16*K bytes: a 128-byte header (the 16 fp32 row scales,
// then zeros) followed by the tile's weights in fragment order -- pairs of
// 16-wide k-steps; inside a pair, 32 lanes x 16 bytes.  Lane l = 4g + t
// holds, per k-step k0, the bytes W[g][k0+2t], W[g][k0+2t+1], W[g+8][k0+2t],
// W[g+8][k0+2t+1], W[g][k0+2t+8], W[g][k0+2t+9], W[g+8][k0+2t+8],
// W[g+8][k0+2t+9], each stored as q + 128.  These are exactly the A-operand
// registers of an m16n8k16 tensor-core MMA, so one 16-byte load feeds two
// MMAs, and a tile is one contiguous run of bytes for a bulk copy.
constexpr int kTileHeader = 128;

// Status word value for a token id outside [0, vocab) met on the device
// (the call reports invalid arguments).
constexpr int kStatusBadToken = 8;
size_t packed_offset(int row, int k, int K);  // byte offset of W[row][k] in the blob sequence
__host__ __device__ inline size_t tile_blob_bytes(int K) { return kTileHeader + 16 * (size_t)K; }

enum GemvMode { kStore = 0, kResid = 1, kSiluGate = 2, kArgmax = 3 };

struct GemvArgs {
    const uint8_t* w;     // tile blobs, rows x K
    const float* scale;   // [rows]
    int rows, K;
    const __half* xh;     // [8*NT][K] f16 planes: column 2b = hi, 2b+1 = lo of sequence b
    int B;                // sequences (<= 4*NT)
    float* y;             // kStore: y[b*ldy + row] = s*acc; kResid: y[b*ldy + row] += s*acc
    int ldy;
    __half* yh;           // kSiluGate: planes [8*NT][ldyh] of a = silu(gate)*up
    int ldyh;
    // kArgmax (lm_head): block-then-grid argmax, lowest index on ties
    unsigned long long* keys;  // [B], zero between launches
    unsigned int* counter;     // zero between launches
    int32_t* tokens;           // [B] next token
    int32_t* out_ids;          // [B][out_cap], column = *step
    int32_t* step;             // device step counter (incremented)
    int out_cap;
    int32_t* pos;              // [B] positions, += 1 when advance_pos
    int advance_pos;
    int valid_rows;            // rows >= valid_rows (padding) take no part in the argmax
    float* logits;             // optional [B][valid_rows]
    int ksplit;                // kResid only: K split over this many CTAs per tile (0 = 1).  The staged
                               // kernel (launch_gemv's choice whenever a CTA's weight slice fits in shared
                               // memory) meets the parts in a thread-block cluster, in rank order.  The
                               // per-item kernel parks them in kpart [tiles][ksplit][4 NT 16] and the last
                               // CTA of a tile (tile_cnt [tiles], zero between launches, left zero) adds
                               // them in order; without kpart each part atomically adds its share to y
    float* kpart;
    unsigned int* tile_cnt;
    int xfrag;                 // xh is in fragment order (plane_index), else plain [8*NT][K] planes
    int yfrag;                 // kSiluGate: yh in fragment order
    // RMSNorm folded into its neighbours.  kResid (staged kernel, or the
    // per-item kernel with kpart): the CTA that finishes a tile also writes
    // the next norm's operand planes, norm_g * x in
    // fragment order (hi/lo), for its rows into norm_xh ([8*NT][norm_H]),
    // and adds its rows' sum of squares of x per sequence to ss_out (64-bit
    // fixed point, value * 2^32: the sum does not depend on the order of the
    // adds).  kStore / kSiluGate / kArgmax: each sequence's dot products are
    // multiplied by 1 / sqrt(ss_in / norm_H + eps) (ss_in NULL: by 1).
    // ss_clear: accumulators [B] that CTA 0 zeroes after the wait, for a
    // later writer.
    const float* norm_g;
    __half* norm_xh;
    long long* ss_out;
    const long long* ss_in;
    long long* ss_clear;
    int norm_H;
    float eps;
    int32_t* status;           // Q3 status word (a bounded wait that ran out), may be null
    // 1: the next kernel may launch only once this one has passed its wait,
    // so that the next kernel's prologue may read what every launch before
    // this one wrote (the decode attention's positions and cached K/V)
    int late_dependents;
};

// Activation planes hold column c = 2b + part (part 0 = f16 hi, 1 = lo of
// sequence b) over K.  Plain order: c * K + k.  Fragment order: the B
// operand registers of the m16n8k16 MMA, so that a lane's four words for
// one k-pair (32 k) and one 8-column tile are one 16-byte load:
// word ((p * 8 + c / 8) * 32 + lane) * 4 + w, lane = 4 (c % 8) + (k % 8) / 2,
// w = 2 ((k / 16) % 2) + (k / 8) % 2, p = k / 32; half k % 2 of the word.
// Room for 8 column tiles (32 sequences), as the plain layout.
__host__ __device__ inline size_t plane_index(int col, int k, int K, int frag) {
    if (!frag) return (size_t)col * K + k;
    const size_t word = (((size_t)(k >> 5) * 8 + (col >> 3)) * 32 + ((col & 7) * 4 + ((k & 7) >> 1))) * 4 +
                        (((k >> 4) & 1) * 2 + ((k >> 3) & 1));
    return word * 2 + (k & 1);
}

// Opts kernel fn in to the device's largest dynamic shared memory on the
// current device, once per (kernel, device); thread-safe.
cudaError_t allow_max_dynamic_smem(const void* fn);

void launch_gemv(const GemvArgs& a, int mode, int grid, cudaStream_t st);
int gemv_grid(int rows, int mode, int num_sms);

// x[r] = float(E[ids[r]]) * sE[ids[r]]; an id outside [0, vocab) gives a zero row and status kStatusBadToken.
void launch_embed(const int32_t* ids, int n, const int8_t* E, const float* sE, int H, int vocab, float* x,
                  int32_t* status, cudaStream_t st);

// RMSNorm of rows (row map optional) -> fp32 rows and/or f16 hi/lo planes.
void launch_rmsnorm(const float* x, const int32_t* rows, int n, int H, const float* g, float eps, float* xn,
                    __half* xh, cudaStream_t st, int frag = 0);

void launch_qk_rope_append(const float* qkv, int R, int nh, int nkv, int hd, const int32_t* row_seq,
                           const int32_t* row_pos, const float* q_norm, const float* k_norm, float eps,
                           const float2* rope_cs, float* q_out, __nv_bfloat16* kc, __nv_bfloat16* vc, int cap,
                           cudaStream_t st);

size_t attn_part_bytes(int R, int nh, int hd, int splits);
// Attends positions 0 .. row_len[r] + len_add - 1 of sequence row_seq[r].
int launch_attention(const float* q, const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* row_seq,
                     const int32_t* row_len, int len_add, int R, int nh, int nkv, int hd, int cap, int splits,
                     float* part, float* out, __half* outh, int ldh, int32_t* status, cudaStream_t st,
                     int frag = 0);

// Decode attention CTAs (head_dim hd, group nh / nkv) resident per SM of the
// current device (0 if the shape is not built or the query failed).
int attention_decode_blocks_per_sm(int hd, int group);

// One decode step's attention with the QK-RMSNorm, RoPE and bf16 KV append
// folded in: qkv [R][(nh + 2 nkv) hd] fp32 as projected, row_pos[r] the new
// position (appended, then attended with positions 0..row_pos[r]); output
// hi/lo f16 planes (outh, ldh, frag as launch_attention).  G CTAs per kv
// head (R <= G, R <= 32) share the rows' positions by the balanced plan:
// row r gets ceil(len_r / P) splits of P positions, P the smallest multiple
// of 64 for which the splits fit in G and no row has more than smax
// (<= 64); part holds [R][nh][smax] partial states.  A row of one split is
// written by the attention itself; a merge kernel follows when G > R.  The
// launch before this one must trigger its dependents only after its own
// wait: the positions and the cached K/V are read before this kernel waits.
// Returns 0, -1 (head_dim / group not built), -2 (launch set-up failed) or
// -3 (sizes out of range).
int launch_attention_decode(const float* qkv, const float* q_norm, const float* k_norm, float eps,
                            const float2* rope_cs, __nv_bfloat16* kc, __nv_bfloat16* vc, const int32_t* row_seq,
                            const int32_t* row_pos, int R, int nh, int nkv, int hd, int cap, int G, int smax,
                            float* part, __half* outh, int ldh, int32_t* status, cudaStream_t st, int frag);

// Causal prefill attention on tensor cores (GROUP == 2, hd == 128): blocks
// of 32 prompt positions of one sequence, {sequence, first position, flat
// row of the sequence's position 0, length}, built by attn_prefill_blocks
// (returns the count; writes at most cap_blocks).  Output: hi/lo f16 planes
// outh[(2r + part) * ldh + head * hd + d].
bool attn_prefill_supported(int nh, int nkv, int hd);
// slots: the KV cache sequence of prompt b (NULL: b itself).
int attn_prefill_blocks(const int32_t* lens, int B, int4* out, int cap_blocks, const int32_t* slots = nullptr);
int launch_attn_prefill(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, const int4* blocks,
                        int nblocks, int nh, int nkv, int hd, int cap, __half* outh, int ldh, cudaStream_t st);

// Prefill projection on tcgen05 tensor cores: Y = s * (x . W^T) over M rows.
// a_planes: [M][2K] f16, row m = hi(m, :) then lo(m, :); w: [N][K] int8
// row-major.  mode kStore: y[m*ldy + n] = ...; kResid: y[...] += ...;
// kSiluGate (fused gate/up rows): hi/lo planes of silu(gate)*up into
// yh[(2m + part) * ldyh + unit].  Needs N % 128 == 0 and K % 64 == 0.
// Returns 0 when launched, < 0 when the arguments do not fit.
bool tc_gemm_supported(int N, int K);
int launch_tc_gemm(const __half* a_planes, const int8_t* w, const float* scale, int M, int N, int K, int mode,
                   float* y, int ldy, __half* yh, int ldyh, int32_t* status, cudaStream_t st, float* work = nullptr,
                   size_t work_bytes = 0, int num_sms = 0);
// K splits launch_tc_gemm uses for this shape on num_sms SMs (1: none), and
// the fp32 workspace they need (0 when none); a split GEMM is two launches
// (the GEMM and the ordered reduction).
int tc_gemm_splits(int M, int N, int K, int num_sms);
size_t tc_gemm_work_bytes(int M, int N, int K, int num_sms);

}  // namespace q3
