// Small-batch decode step: two kernels per layer plus the lm_head sweep (sm_103a).
//
// The decoder block is the Qwen3 family's ("Model-agnostic LLM inference",
// section "Supported models"): RMSNorm -> QKV -> per-head RMSNorm on Q and
// K -> RoPE -> bf16 KV append -> grouped-query attention -> O + residual ->
// RMSNorm -> SiLU-gated FFN + residual; then the final RMSNorm and the tied
// lm_head with the greedy argmax ("Run local LLM decode", section
// "Limitations").  Single-stream decode streams every weight once per step
// ("LLM inference overview", section "Workload characteristics"), so each
// kernel moves its weights into shared memory before it waits on the
// previous kernel: after the wait only the activations are loaded.
//
// Every kernel is launched with programmatic dependent launch.  A kernel
// lets its successor start only after its own wait has returned, so when a
// kernel's prologue runs, every kernel two or more places before it in the
// stream has completed: the prologues read only constant data (weights,
// scales) and, from the second layer on, the positions and the cached K/V
// of earlier steps.
#include <algorithm>

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "step.h"

namespace cg = cooperative_groups;

namespace q3 {
namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr int kWarps = 8;
constexpr int kLmThreads = 288;  // lm_head: up to 8 consumer warps + 1 producer warp

// ------------------------------------------------------------- fixed point
// The residual stream between kernels is value * 2^32 in a signed 64-bit
// integer (resolution 2.3e-10, range +-2.1e9).  Partial sums of a split
// projection are converted once and meet in integer atomic adds, which give
// the same bits in any order.
constexpr float kFixOne = 4294967296.0f;
constexpr float kFixUnit = 2.3283064365386963e-10f;

// Both conversions go through 32-bit halves: the 64-bit integer <-> float
// conversions are much slower on this part, and these give the same results
// (round to nearest even into the fixed point; correctly rounded back).
Q3_DEV long long fix_of(float v) {
    const float f = v * kFixOne;
    const float a = fabsf(f);
    const uint32_t hi = __float2uint_rz(a * kFixUnit);
    const float rem = a - (float)hi * kFixOne;  // exact: a multiple of ulp(a) below 2^32
    const unsigned long long m = ((unsigned long long)hi << 32) + __float2uint_rn(rem);
    return f < 0.f ? -(long long)m : (long long)m;
}
Q3_DEV float float_of_fix(long long x) {
    const bool neg = x < 0;
    const unsigned long long m = neg ? (unsigned long long)(-(x + 1)) + 1ull : (unsigned long long)x;
    const float v = __uint2float_rn((uint32_t)(m >> 32)) + __uint2float_rn((uint32_t)m) * kFixUnit;
    return neg ? -v : v;
}
Q3_DEV void red_add_fix(long long* p, long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ------------------------------------------------------------- operands
// Index of the f16 half for column col (0..7) and k within one 8-column tile
// of a fragment-ordered B operand (the m16n8k16 B registers of lane
// 4 col + (k % 8) / 2, word 2 ((k / 16) % 2) + (k / 8) % 2, half k % 2).
Q3_DEV int frag_half(int col, int k) {
    const int lanef = col * 4 + ((k & 7) >> 1);
    const int w = ((k >> 4) & 1) * 2 + ((k >> 3) & 1);
    return (((k >> 5) * 32 + lanef) * 4 + w) * 2 + (k & 1);
}

Q3_DEV uint32_t pack_half2(__half a, __half b) {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

// 32-bit word of the fragment-ordered B operand (one 8-column tile) that
// holds column col, k and k + 1 (k even).
Q3_DEV int frag_word(int col, int k) {
    return (((k >> 5) * 32 + col * 4 + ((k & 7) >> 1)) * 4) + ((k >> 4) & 1) * 2 + ((k >> 3) & 1);
}

// RMSNorm of up to 4 rows into the fragment-ordered B operand of one 8-column
// MMA tile: column 2b holds f16(v) and column 2b + 1 holds f16(v - f16(v)) of
// v = (x[b][k] * inv_rms[b]) * gain[k].  Columns of rows b >= B are left
// as they are: each output column of an MMA depends only on its own operand
// column, so those outputs are simply never read.  x is read from the
// fixed-point stream xin ([B][H]) or, with xin null, is the embedding row of
// token tok[b] (emb, emb_scale); gain is in shared memory.  Thread t owns
// k = 4t .. 4t + 3; every thread of the block takes part in the barriers.
// H <= 4 * 256.
Q3_DEV void norm_operand(uint4* xop, const long long* xin, const int* tok, const int8_t* emb, const float* emb_scale,
                         int B, int H, const float* gain, float eps, float* s_red) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool own = tid < kThreads && 4 * tid < H;
    const int k0 = 4 * tid;
    float x[kStepMaxBatch][4];
    float ss[kStepMaxBatch];
#pragma unroll
    for (int b = 0; b < kStepMaxBatch; ++b) {
        ss[b] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) x[b][j] = 0.f;
        if (own && b < B) {
            if (xin) {
                const longlong2 v0 = __ldcg(reinterpret_cast<const longlong2*>(xin + (size_t)b * H + k0));
                const longlong2 v1 = __ldcg(reinterpret_cast<const longlong2*>(xin + (size_t)b * H + k0 + 2));
                x[b][0] = float_of_fix(v0.x), x[b][1] = float_of_fix(v0.y);
                x[b][2] = float_of_fix(v1.x), x[b][3] = float_of_fix(v1.y);
            } else {
                const int t = tok[b];
                const char4 e = *reinterpret_cast<const char4*>(emb + (size_t)t * H + k0);
                const float es = emb_scale[t];
                x[b][0] = (float)e.x * es, x[b][1] = (float)e.y * es, x[b][2] = (float)e.z * es, x[b][3] = (float)e.w * es;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) ss[b] += x[b][j] * x[b][j];
        }
    }
#pragma unroll
    for (int b = 0; b < kStepMaxBatch; ++b)
        if (b < B) {
            ss[b] = warp_sum(ss[b]);
            if (lane == 0 && warp < kWarps) s_red[warp * 4 + b] = ss[b];
        }
    __syncthreads();
    if (own) {
        const float4 g = *reinterpret_cast<const float4*>(gain + k0);
        const float gg[4] = {g.x, g.y, g.z, g.w};
        uint32_t* xw = reinterpret_cast<uint32_t*>(xop);
#pragma unroll
        for (int b = 0; b < kStepMaxBatch; ++b) {
            if (b >= B) break;
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t += s_red[w * 4 + b];
            const float inv = 1.0f / sqrtf(t / (float)H + eps);
            __half hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) split_f16(__fmul_rn(__fmul_rn(x[b][j], inv), gg[j]), hi[j], lo[j]);
            xw[frag_word(2 * b, k0)] = pack_half2(hi[0], hi[1]);
            xw[frag_word(2 * b, k0 + 2)] = pack_half2(hi[2], hi[3]);
            xw[frag_word(2 * b + 1, k0)] = pack_half2(lo[0], lo[1]);
            xw[frag_word(2 * b + 1, k0 + 2)] = pack_half2(lo[2], lo[3]);
        }
    }
    __syncthreads();
}

// Two m16n8k16 MMAs from one 16-byte lane chunk of a tile blob (rows g, g+8;
// two 16-wide k-steps) and the lane's four B words; the weights are
// converted exactly (byte permute and subtraction of the 128 offset).
Q3_DEV void mma_pair(float (&c0)[4], float (&c1)[4], const uint4& wv, const uint4& bv) {
    uint32_t A0[4], A1[4];
    u8x4_to_f16x2x2(wv.x, A0[0], A0[1]);
    u8x4_to_f16x2x2(wv.y, A0[2], A0[3]);
    u8x4_to_f16x2x2(wv.z, A1[0], A1[1]);
    u8x4_to_f16x2x2(wv.w, A1[2], A1[3]);
    mma_f16_16816(c0, A0, bv.x, bv.y);
    mma_f16_16816(c1, A1, bv.z, bv.w);
}

// mbar_wait_bounded with its polling loop out of line: one try inline (the
// common case, the phase has completed or completes within the try's own
// suspend window), the loop only when that try fails.  Keeps the kernels'
// code, fetched once per launch, small.
__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity) { return mbar_wait_bounded(bar, parity); }
Q3_DEV bool wait_phase(uint64_t* bar, uint32_t parity) { return mbar_try_wait(bar, parity) || wait_slow(bar, parity); }

// Bounded wait shared by a whole block: every thread waits, and the block
// agrees on the outcome (true when any thread's wait gave up).
Q3_DEV bool block_wait_failed(uint64_t* bar, uint32_t parity) {
    const bool ok = wait_phase(bar, parity);
    return __syncthreads_or(!ok) != 0;
}

// The operand of one K slice.  Columns 2b and 2b + 1 hold f16(v) and
// f16(v - f16(v)) of v = gain[k] * x[b][k] for the slice's local k = 0 ..
// 32 nkp - 1 (global k = kbase + local); the RMSNorm's 1 / rms is a factor of
// the whole row and is applied to the finished dot products instead.
// s_ss[b] receives the slice's sum of squares of x[b].  x comes from the
// fixed-point stream xin ([B][H]) or, with xin null, is the embedding row of
// token tok[b].  Thread t < 8 nkp B owns 4 consecutive k of sequence
// t / (8 nkp); 8 nkp <= 32, so a sequence's threads share one warp.
Q3_DEV void slice_operand(uint4* xop, float* s_ss, const long long* xin, const int* tok, const int8_t* emb,
                          const float* emb_scale, int B, int H, int kbase, int nkp, const float* s_gain) {
    const int t = threadIdx.x;
    const int per_b = 8 * nkp;
    const bool own = t < B * per_b;
    const int b = own ? t / per_b : 0;
    const int kl = 4 * (t - b * per_b);
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (own) {
        const int k = kbase + kl;
        if (xin) {
            const longlong2 v0 = __ldcg(reinterpret_cast<const longlong2*>(xin + (size_t)b * H + k));
            const longlong2 v1 = __ldcg(reinterpret_cast<const longlong2*>(xin + (size_t)b * H + k + 2));
            x[0] = float_of_fix(v0.x), x[1] = float_of_fix(v0.y), x[2] = float_of_fix(v1.x), x[3] = float_of_fix(v1.y);
        } else {
            const int tk = tok[b];
            const char4 e = *reinterpret_cast<const char4*>(emb + (size_t)tk * H + k);
            const float es = emb_scale[tk];
            x[0] = (float)e.x * es, x[1] = (float)e.y * es, x[2] = (float)e.z * es, x[3] = (float)e.w * es;
        }
    }
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    __half hi[4], lo[4];
    {
        const float4 g = own ? *reinterpret_cast<const float4*>(s_gain + kl) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float gg[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) split_f16(__fmul_rn(gg[j], x[j]), hi[j], lo[j]);
    }
    // sum over the per_b threads of this sequence (an aligned group inside one warp)
    for (int o = 1; o < per_b; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (own) {
        if (kl == 0) s_ss[b] = ss;
        uint32_t* xw = reinterpret_cast<uint32_t*>(xop);
        xw[frag_word(2 * b, kl)] = pack_half2(hi[0], hi[1]);
        xw[frag_word(2 * b, kl + 2)] = pack_half2(hi[2], hi[3]);
        xw[frag_word(2 * b + 1, kl)] = pack_half2(lo[0], lo[1]);
        xw[frag_word(2 * b + 1, kl + 2)] = pack_half2(lo[2], lo[3]);
    }
}

// Partial sums of a cluster's tiles over this CTA's K slice: warp w takes
// tiles w, w + 8, ... (< nt) of the slice blobs at w_slices (nkp k-pairs,
// 512 bytes each, per tile) against the slice operand, and writes row
// 16 t + g (and + 8) of sequence column q to out[q * ld + row], q = 0..3
// (the columns of absent sequences hold whatever their operand columns gave).
template <int TPW>
Q3_DEV void cluster_tiles_mma(const unsigned char* w_slices, int nt, int nkp, const uint4* xop, float* out, int ld) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    float c0[TPW][4], c1[TPW][4];
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) c0[i][e] = c1[i][e] = 0.f;
    for (int p = 0; p < nkp; ++p) {
        const uint4 bv = xop[p * 32 + lane];
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
            const int t = warp + kWarps * i;
            if (t < nt) {
                const uint4 wv = *reinterpret_cast<const uint4*>(w_slices + ((size_t)t * nkp + p) * 512 + lane * 16);
                mma_pair(c0[i], c1[i], wv, bv);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
        const int t = warp + kWarps * i;
        if (t < nt) {
            out[q * ld + t * 16 + g] = c0[i][0] + c0[i][1] + c1[i][0] + c1[i][1];
            out[q * ld + t * 16 + g + 8] = c0[i][2] + c0[i][3] + c1[i][2] + c1[i][3];
        }
    }
}

// Sum over the 8 CTAs of a cluster of element i of a shared array, as a
// fixed pairwise tree (every CTA gets the same bits).
Q3_DEV float cluster_sum(const float* arr, int i) {
    float v[kClusterCtas];
#pragma unroll
    for (int r = 0; r < kClusterCtas; ++r) v[r] = peer(arr, r)[i];
    return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

// 1 / rms of sequence b from the cluster's partial sums of squares (s_ss of
// slice_operand).
Q3_DEV float cluster_inv_rms(const float* s_ss, int b, int H, float eps) {
    return 1.0f / sqrtf(cluster_sum(s_ss, b) / (float)H + eps);
}

// Clears this CTA's share of a [n] accumulator (fire-and-forget stores).
Q3_DEV void clear_share(long long* p, int n) {
    if (!p) return;
    const int per = (n + gridDim.x - 1) / gridDim.x;
    const int z0 = blockIdx.x * per, z1 = min(n, z0 + per);
#pragma unroll 1
    for (int i = z0 + (int)threadIdx.x; i < z1; i += blockDim.x) p[i] = 0;
}

}  // namespace

// ===================================================================== layouts
__host__ __device__ inline uint32_t take_smem(uint32_t& off, size_t bytes) {
    const uint32_t o = off;
    off = (uint32_t)((off + bytes + 127) & ~(size_t)127);
    return o;
}

struct AttnBlockLayout {
    uint32_t wq, qn, kn, vn, wst, part, oop, wo, xop, pqkv, ss, ring, sc, osc, gain, qkg, rope, resid, misc, bars, total;
};

// The QKV weight slices are dead once the partial sums are written: the
// per-head vectors, the softmax states and the O operand reuse that region.
__host__ __device__ inline AttnBlockLayout attn_block_layout(int H, int hd, int kv_stages) {
    AttnBlockLayout L{};
    uint32_t off = 0;
    const int T = 3 * hd / 16, nkp = H / 32 / kClusterCtas;
    {
        uint32_t w = 0;
        L.qn = take_smem(w, (size_t)kStepMaxBatch * hd * 4);
        L.kn = take_smem(w, (size_t)kStepMaxBatch * hd * 4);
        L.vn = take_smem(w, (size_t)kStepMaxBatch * hd * 4);
        L.wst = take_smem(w, (size_t)kWarps * kStepMaxBatch * (hd + 4) * 4);  // warp states, then the parked parts
        L.part = take_smem(w, (size_t)kStepMaxBatch * (hd + 4) * 4);    // 16-byte aligned states
        L.oop = take_smem(w, (size_t)(hd / 32) * 512);
        const size_t wq_bytes = (size_t)T * nkp * 512;
        L.wq = take_smem(off, wq_bytes > w ? wq_bytes : w);
        L.qn += L.wq, L.kn += L.wq, L.vn += L.wq, L.wst += L.wq, L.part += L.wq, L.oop += L.wq;
    }
    L.wo = take_smem(off, (size_t)(H / kClusterCtas / 16) * (hd / 32) * 512);
    L.xop = take_smem(off, (size_t)nkp * 512);
    L.pqkv = take_smem(off, (size_t)kStepMaxBatch * 3 * hd * 4);
    L.ss = take_smem(off, (size_t)kStepMaxBatch * 4);
    L.ring = take_smem(off, (size_t)kv_stages * 2 * kStepKvChunk * hd * 2);
    L.sc = take_smem(off, (size_t)3 * hd * 4);
    L.osc = take_smem(off, (size_t)(H / kClusterCtas) * 4);
    L.gain = take_smem(off, (size_t)nkp * 32 * 4);
    L.qkg = take_smem(off, (size_t)2 * hd * 4);
    L.rope = take_smem(off, (size_t)kStepMaxBatch * (hd / 2) * 8);
    L.resid = take_smem(off, (size_t)kStepMaxBatch * (H / kClusterCtas) * 8);
    L.misc = take_smem(off, 256);
    L.bars = take_smem(off, (size_t)(2 + kv_stages) * 8);
    L.total = off;
    return L;
}

struct FfnLayout {
    uint32_t wgu, wd, xop, dop, sgu, sd, red, resid, bars, total;
};
__host__ __device__ inline FfnLayout ffn_layout(int H) {
    FfnLayout L{};
    uint32_t off = 0;
    L.wgu = take_smem(off, (size_t)(2 * kFfnUnits / 16) * tile_blob_bytes(H));
    L.wd = take_smem(off, (size_t)(H / 16) * 512);
    // the operand, then the warps' partial gate/up rows
    const size_t part = (size_t)kWarps * kStepMaxBatch * 2 * kFfnUnits * 4, xop = (size_t)(H / 32) * 512;
    L.xop = take_smem(off, xop > part ? xop : part);
    L.dop = take_smem(off, 512);
    L.sgu = take_smem(off, (size_t)2 * kFfnUnits * 4);
    L.sd = take_smem(off, (size_t)H * 4);
    L.red = take_smem(off, (size_t)kWarps * 4 * 4);
    L.resid = take_smem(off, (size_t)kStepMaxBatch * kFfnResidRows * 8);
    L.bars = take_smem(off, 2 * 8);
    L.total = off;
    return L;
}

struct LmLayout {
    uint32_t ring, xop, gain, best, misc, bars, total;
};
__host__ __device__ inline LmLayout lm_layout(int H, int stages) {
    LmLayout L{};
    uint32_t off = 0;
    L.ring = take_smem(off, (size_t)stages * tile_blob_bytes(H));
    L.xop = take_smem(off, (size_t)(H / 32) * 512);
    L.gain = take_smem(off, (size_t)H * 4);
    L.best = take_smem(off, (size_t)kWarps * 4 * 8);
    L.misc = take_smem(off, 512);
    L.bars = take_smem(off, (size_t)2 * stages * 8);
    L.total = off;
    return L;
}

// ===================================================================== attention block
// Cluster h (8 CTAs) serves query head h of kv group g = h / (nh / nkv).
//  1. The cluster's QKV rows (head h of Wq, group g of Wk and Wv: 3 hd rows
//     in 16-row tiles) are multiplied by the residual stream, K split over the
//     8 CTAs: CTA r holds the k-pairs [r KP / 8, (r + 1) KP / 8) of every
//     tile in shared memory and warp w the tiles w, w + 8, ...; the RMSNorm
//     gain is folded into the operand and 1 / rms into the result.
//  2. Every CTA sums the 8 partial rows (distributed shared memory) for the
//     vectors it needs, applies the row scales, 1 / rms, the per-head RMSNorm
//     of q and k and RoPE at the sequence's position, and rounds k and v to
//     bf16.  CTA 7 of the group's first cluster appends them to the cache
//     (at the very end, so that no barrier waits for those stores).
//  3. The cached positions 0..p-1 of each sequence are split over the 8 CTAs
//     (16-position chunks staged by bulk copies); CTA 7 also attends the new
//     position p from the rounded values.  Each CTA keeps an online softmax
//     state (m, l, acc) per sequence.
//  4. Every CTA merges the 8 states into the head's output o and multiplies
//     its H / 8 rows of Wo[:, head h] by it; the rows are added to the
//     fixed-point residual stream (cluster 0 also adds the stream's input).
// Before the wait the CTA starts the bulk copies of its weight slices and O
// rows and copies the gains, row scales and (from the second layer on,
// where the positions are final) the RoPE rows into shared memory and starts
// its K/V stages; after the wait the only global reads are its slice of the
// residual rows (in the first layer: the tokens and their embedding).
template <int HD>
__global__ void __launch_bounds__(kThreads, 2) attn_block_kernel(const AttnBlockArgs a) {
    constexpr int D = HD / 32;  // elements per lane of a head vector (lane l: D l .. D l + D - 1)
    constexpr int TH = HD / 16;
    constexpr int T = 3 * TH;
    constexpr int TPW = (T + kWarps - 1) / kWarps;
    constexpr int PS = HD + 4;  // floats per softmax state {acc[HD], m, l, pad}: 16-byte aligned rows
    constexpr int R3 = 3 * HD;  // rows of the cluster
    extern __shared__ __align__(128) unsigned char smem[];
    const AttnBlockLayout L = attn_block_layout(a.H, HD, a.kv_stages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = cluster_rank();
    const int h = blockIdx.x / kClusterCtas;
    const int G = a.nh / a.nkv, g = h / G;
    const int H = a.H, B = a.B, S = a.kv_stages;
    const int Dq = a.nh * HD, Dkv = a.nkv * HD;
    const int nkp = H / 32 / kClusterCtas, kp0 = r * nkp;
    const uint32_t blob = (uint32_t)tile_blob_bytes(H);
    const int ro = H / kClusterCtas, otiles = ro / 16;
    const uint32_t oseg = (HD / 32) * 512;
    const uint32_t oblob = (uint32_t)tile_blob_bytes(Dq);
    const bool appender = (h % G == 0) && (r == kClusterCtas - 1);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);  // 0 QKV slices, 1 O rows, 2.. K/V stages
    int* s_pos = reinterpret_cast<int*>(smem + L.misc);
    int* s_seq = s_pos + 4;
    int* s_tok = s_seq + 4;
    int* s_last = s_tok + 4;  // [S] last item issued into each stage (-1: none)
    float* s_sc = reinterpret_cast<float*>(smem + L.sc);
    float* osc = reinterpret_cast<float*>(smem + L.osc);
    float* s_gain = reinterpret_cast<float*>(smem + L.gain);
    float* s_qg = reinterpret_cast<float*>(smem + L.qkg);
    float* s_kg = s_qg + HD;
    float2* s_rope = reinterpret_cast<float2*>(smem + L.rope);
    long long* s_res = reinterpret_cast<long long*>(smem + L.resid);
    uint4* xop = reinterpret_cast<uint4*>(smem + L.xop);
    float* pqkv = reinterpret_cast<float*>(smem + L.pqkv);
    float* s_ss = reinterpret_cast<float*>(smem + L.ss);
    float* qn = reinterpret_cast<float*>(smem + L.qn);
    float* kn = reinterpret_cast<float*>(smem + L.kn);
    float* vn = reinterpret_cast<float*>(smem + L.vn);
    float* wst = reinterpret_cast<float*>(smem + L.wst);
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint4* oop = reinterpret_cast<uint4*>(smem + L.oop);
    __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem + L.ring);

    auto grow = [&](int j) -> int {  // global QKV row of cluster row j
        if (j < HD) return h * HD + j;
        if (j < 2 * HD) return Dq + g * HD + (j - HD);
        return Dq + Dkv + g * HD + (j - 2 * HD);
    };
    auto o_src = [&](int i) -> const uint8_t* {
        return a.wo + (size_t)(r * otiles + i) * oblob + kTileHeader + (size_t)h * oseg;
    };
    auto split_lo = [&](int b) { return r * s_pos[b] / kClusterCtas; };
    auto split_hi = [&](int b) { return (r + 1) * s_pos[b] / kClusterCtas; };
    auto nchunks = [&](int b) { return (split_hi(b) - split_lo(b) + kStepKvChunk - 1) / kStepKvChunk; };
    auto count_items = [&]() {
        int n = 0;
        #pragma unroll 1
        for (int b = 0; b < B; ++b) n += nchunks(b);
        return n;
    };
    auto issue_kv = [&](int i) {  // thread 0 only
        int b = 0, c = i;
        while (c >= nchunks(b)) c -= nchunks(b), ++b;
        const int lo = split_lo(b) + c * kStepKvChunk;
        const int cnt = min(kStepKvChunk, split_hi(b) - lo);
        const size_t base = (((size_t)s_seq[b] * a.nkv + g) * a.cap + lo) * HD;
        const uint32_t bytes = (uint32_t)cnt * HD * 2u;
        const int s = i % S;
        __nv_bfloat16* dk = ring + (size_t)s * 2 * kStepKvChunk * HD;
        mbar_arrive_expect_tx(&bars[2 + s], 2 * bytes);
        bulk_g2s(dk, a.kc + base, bytes, &bars[2 + s]);
        bulk_g2s(dk + kStepKvChunk * HD, a.vc + base, bytes, &bars[2 + s]);
        s_last[s] = i;
    };
    // positions known: RoPE rows into shared memory; the first K/V stages
    auto position_work = [&]() {
        #pragma unroll 1
        for (int i = tid; i < B * (HD / 2); i += kThreads) {
            const int b = i / (HD / 2), j = i - b * (HD / 2);
            s_rope[i] = a.rope[(size_t)s_pos[b] * (HD / 2) + j];
        }
        if (tid == 0) {
            const int n = count_items();
            #pragma unroll 1
            for (int i = 0; i < S && i < n; ++i) issue_kv(i);
        }
    };

    // ---- prologue: constant data and, from the second layer on, the positions
    if (tid == 0) {
        #pragma unroll 1
        for (int i = 0; i < 2 + S; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        #pragma unroll 1
        for (int i = 0; i < S; ++i) s_last[i] = -1;
    }
    if (a.pos_early && tid < B) {
        s_pos[tid] = a.pos[tid];
        s_seq[tid] = a.seq_ids[tid];
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], (uint32_t)(T * nkp * 512));
        #pragma unroll 1
        for (int t = 0; t < T; ++t)
            bulk_g2s(smem + L.wq + (size_t)t * nkp * 512,
                     a.wqkv + (size_t)(grow(t * 16) / 16) * blob + kTileHeader + (size_t)kp0 * 512,
                     (uint32_t)nkp * 512, &bars[0]);
        mbar_arrive_expect_tx(&bars[1], (uint32_t)otiles * oseg);
        #pragma unroll 1
        for (int i = 0; i < otiles; ++i) bulk_g2s(smem + L.wo + (size_t)i * oseg, o_src(i), oseg, &bars[1]);
    }
    #pragma unroll 1
    for (int i = tid; i < R3; i += kThreads) s_sc[i] = a.qkv_scale[grow(i)];
    #pragma unroll 1
    for (int i = tid; i < ro; i += kThreads) osc[i] = a.o_scale[r * ro + i];
    #pragma unroll 1
    for (int i = tid; i < nkp * 32; i += kThreads) s_gain[i] = a.attn_norm[kp0 * 32 + i];
    #pragma unroll 1
    for (int i = tid; i < HD; i += kThreads) s_qg[i] = a.q_norm[i], s_kg[i] = a.k_norm[i];
    if (a.pos_early) position_work();
    pdl_wait();
    pdl_launch_dependents();

    // ---- after the wait: positions and tokens (first layer), residual rows, accumulators to clear
    if (!a.pos_early) {
        if (tid < B) {
            s_pos[tid] = a.pos[tid];
            s_seq[tid] = a.seq_ids[tid];
            if (!a.xin) {
                // a token outside the table is never dereferenced: it reads row 0 and the call reports it
                const int t = a.tokens[tid];
                const bool okt = t >= 0 && t < a.vocab;
                if (!okt) set_status(a.status, kStatusBadToken);
                s_tok[tid] = okt ? t : 0;
            }
        }
        __syncthreads();
        position_work();
    }
    if (h == 0)  // this cluster adds the stream's input to its rows
        #pragma unroll 1
        for (int i = tid; i < B * ro; i += kThreads) {
            const int b = i / ro, R = r * ro + (i - b * ro);
            s_res[i] = a.xin ? __ldcg(a.xin + (size_t)b * H + R)
                             : fix_of((float)a.emb[(size_t)s_tok[b] * H + R] * a.emb_scale[s_tok[b]]);
        }
    clear_share(a.clear0, B * H);
    clear_share(a.clear1, B * H);
    const int n_items = count_items();

    // ---- 1. this CTA's K slice of the cluster's QKV rows
    slice_operand(xop, s_ss, a.xin, s_tok, a.emb, a.emb_scale, B, H, kp0 * 32, nkp, s_gain);
    bool bad = block_wait_failed(&bars[0], 0);
    if (!bad) cluster_tiles_mma<TPW>(smem + L.wq, T, nkp, xop, pqkv, R3);
    cluster_arrive();
    cluster_wait();  // every CTA's partial rows are visible in the cluster

    // ---- 2. q, k, v of each sequence: partial rows summed, scaled, normed, rotated
    // warp b < B: query of sequence b; warp 4 + b: key and value of sequence b.
    // Lane l holds elements D l .. D l + D - 1; the RoPE partner of element i
    // (i + hd / 2 or i - hd / 2) sits in lane l ^ 16.
    if ((warp & 3) < B) {
        const int b = warp & 3;
        const bool is_q = warp < 4;
        const float inv = cluster_inv_rms(s_ss, b, H, a.eps);
        // v = scale * inv * (sum over the peers), rows j0 + D l .. (pairwise tree over the peers)
        auto rows = [&](int j0, float (&v)[D]) {
            float pr[kClusterCtas][D];
#pragma unroll
            for (int rr = 0; rr < kClusterCtas; ++rr) {
                const float* pp = peer(pqkv, rr) + b * R3 + j0 + D * lane;
                if constexpr (D == 4) {
                    const float4 x = *reinterpret_cast<const float4*>(pp);
                    pr[rr][0] = x.x, pr[rr][1] = x.y, pr[rr][2] = x.z, pr[rr][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2*>(pp);
                    pr[rr][0] = x.x, pr[rr][1] = x.y;
                }
            }
#pragma unroll
            for (int m = 0; m < D; ++m) {
                const float t = ((pr[0][m] + pr[1][m]) + (pr[2][m] + pr[3][m])) +
                                ((pr[4][m] + pr[5][m]) + (pr[6][m] + pr[7][m]));
                v[m] = s_sc[j0 + D * lane + m] * inv * t;
            }
        };
        float v[D], vv[D];
        rows(is_q ? 0 : HD, v);
        if (!is_q) rows(2 * HD, vv);
        const float* gain = is_q ? s_qg : s_kg;
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < D; ++m) ss += v[m] * v[m];
        ss = warp_sum(ss);
        const float hinv = 1.0f / sqrtf(ss / (float)HD + a.eps);
#pragma unroll
        for (int m = 0; m < D; ++m) v[m] = __fmul_rn(__fmul_rn(v[m], hinv), gain[D * lane + m]);
        const float2* cs = s_rope + b * (HD / 2) + D * (lane & 15);
#pragma unroll
        for (int m = 0; m < D; ++m) {
            const float pv = __shfl_xor_sync(0xffffffffu, v[m], 16);
            const float2 c = cs[m];
            v[m] = lane < 16 ? __fsub_rn(__fmul_rn(v[m], c.x), __fmul_rn(pv, c.y))
                             : __fadd_rn(__fmul_rn(v[m], c.x), __fmul_rn(pv, c.y));
        }
#pragma unroll
        for (int m = 0; m < D; ++m) {
            if (is_q) {
                qn[b * HD + D * lane + m] = v[m];
            } else {
                kn[b * HD + D * lane + m] = __bfloat162float(__float2bfloat16_rn(v[m]));
                vn[b * HD + D * lane + m] = __bfloat162float(__float2bfloat16_rn(vv[m]));
            }
        }
    }
    __syncthreads();

    // ---- 3. attention over this CTA's split of every sequence
    const float scale = 1.0f / sqrtf((float)HD);
    int item = 0;
    for (int b = 0; b < B; ++b) {
        float q[D], acc[D];
        float m = -INFINITY, l = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) q[d] = qn[b * HD + lane * D + d], acc[d] = 0.f;
        const int lo = split_lo(b), hi = split_hi(b), nch = nchunks(b);
        for (int c = 0; c < nch; ++c, ++item) {
            const int s = item % S;
            const bool ok = bad || wait_phase(&bars[2 + s], (uint32_t)(item / S) & 1u);
            const int cnt = min(kStepKvChunk, hi - lo - c * kStepKvChunk);
            const __nv_bfloat16* ks = ring + (size_t)s * 2 * kStepKvChunk * HD;
            const __nv_bfloat16* vs = ks + kStepKvChunk * HD;
            float sc[kStepKvChunk / kWarps];
#pragma unroll
            for (int i = 0; i < kStepKvChunk / kWarps; ++i) {
                const int j = warp + kWarps * i;
                float dot = 0.f;
                if (j < cnt && ok && !bad) {
                    const __nv_bfloat16* kr = ks + (size_t)j * HD + lane * D;
#pragma unroll
                    for (int d = 0; d < D; ++d) dot += q[d] * __bfloat162float(kr[d]);
                }
                dot = warp_sum(dot);
                sc[i] = (j < cnt) ? dot * scale : -INFINITY;
            }
            float cm = sc[0];
#pragma unroll
            for (int i = 1; i < kStepKvChunk / kWarps; ++i) cm = fmaxf(cm, sc[i]);
            const float mn = fmaxf(m, cm);
            if (mn != -INFINITY) {
                const float corr = (m == -INFINITY) ? 0.f : expf(m - mn);
                l *= corr;
#pragma unroll
                for (int d = 0; d < D; ++d) acc[d] *= corr;
#pragma unroll
                for (int i = 0; i < kStepKvChunk / kWarps; ++i) {
                    if (sc[i] == -INFINITY) continue;
                    const float p = expf(sc[i] - mn);
                    l += p;
                    const __nv_bfloat16* vr = vs + (size_t)(warp + kWarps * i) * HD + lane * D;
#pragma unroll
                    for (int d = 0; d < D; ++d) acc[d] += p * __bfloat162float(vr[d]);
                }
                m = mn;
            }
            bad = __syncthreads_or(!ok) != 0 || bad;  // every warp is done with stage s
            if (tid == 0 && !bad && item + S < n_items) issue_kv(item + S);
        }
        if (r == kClusterCtas - 1 && warp == 0) {
            // the new position, from the rounded values in shared memory
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < D; ++d) dot += q[d] * kn[b * HD + lane * D + d];
            const float sc = warp_sum(dot) * scale;
            const float mn = fmaxf(m, sc);
            const float corr = (m == -INFINITY) ? 0.f : expf(m - mn);
            const float pe = expf(sc - mn);
            l = l * corr + pe;
#pragma unroll
            for (int d = 0; d < D; ++d) acc[d] = acc[d] * corr + pe * vn[b * HD + lane * D + d];
            m = mn;
        }
        // park this warp's state for sequence b (merged once for every sequence below)
        float* ws = wst + (b * kWarps + warp) * PS;
        if (lane == 0) ws[HD] = m, ws[HD + 1] = l;
#pragma unroll
        for (int d = 0; d < D; ++d) ws[lane * D + d] = acc[d];
    }
    __syncthreads();
    // merge the 8 warps' states of each sequence into this CTA's state: the
    // thread of element (b, d) derives the warps' weights from their (m, l)
    // in warp order and sums its element
#pragma unroll 1
    for (int i = tid; i < B * HD; i += kThreads) {
        const int b = i / HD, d = i - b * HD;
        const float* wb = wst + b * kWarps * PS;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wb[w * PS + HD]);
        float Ls = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = wb[w * PS + HD];
            const float f = (mw == -INFINITY) ? 0.f : expf(mw - M);
            Ls += wb[w * PS + HD + 1] * f;
            A += wb[w * PS + d] * f;
        }
        float* pb = part + b * PS;
        pb[d] = A;
        if (d == 0) pb[HD] = M, pb[HD + 1] = Ls;
    }
    __syncthreads();

    // ---- 4. merge the cluster's states; this CTA's rows of Wo[:, head h]
    cluster_arrive();
    cluster_wait();  // every CTA's states are visible in the cluster
    {
        // warp w scales CTA w's state by its softmax weight (every warp
        // derives the same weights from the 8 (m, l) pairs) and parks it;
        // each output element then sums the 8 parked parts in rank order
        float* contrib = wst;  // [8][4][HD] (the warps' states are merged)
        const float* mine = peer(part, warp);
#pragma unroll
        for (int b = 0; b < kStepMaxBatch; ++b) {
            if (b >= B) break;
            const float mr = lane < kClusterCtas ? peer(part, lane)[b * PS + HD] : -INFINITY;
            const float lr = lane < kClusterCtas ? peer(part, lane)[b * PS + HD + 1] : 0.f;
            const float M = warp_max(mr);
            const float f = mr == -INFINITY ? 0.f : expf(mr - M);
            const float Ls = warp_sum(lr * f);
            const float fw = __shfl_sync(0xffffffffu, f, warp) / Ls;
            if (lane < HD / 4) {
                const float4 x = *reinterpret_cast<const float4*>(mine + b * PS + lane * 4);
                *reinterpret_cast<float4*>(contrib + (warp * kStepMaxBatch + b) * HD + lane * 4) =
                    make_float4(x.x * fw, x.y * fw, x.z * fw, x.w * fw);
            }
        }
        __syncthreads();
        __half* ooph = reinterpret_cast<__half*>(oop);
        #pragma unroll 1
        for (int i = tid; i < B * HD; i += kThreads) {
            const int b = i / HD, d = i - b * HD;
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kClusterCtas; ++w) o += contrib[(w * kStepMaxBatch + b) * HD + d];
            __half hi, lo;
            split_f16(o, hi, lo);
            ooph[frag_half(2 * b, d)] = hi;
            ooph[frag_half(2 * b + 1, d)] = lo;
        }
    }
    cluster_arrive();  // done with the peers' shared memory (waited for before leaving)
    bad = block_wait_failed(&bars[1], 0) || bad;
    if (warp < otiles && !bad) {
        const unsigned char* wt = smem + L.wo + (size_t)warp * oseg;
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < HD / 32; ++p) {
            const uint4 wv = *reinterpret_cast<const uint4*>(wt + p * 512 + lane * 16);
            mma_pair(c0, c1, wv, oop[p * 32 + lane]);
        }
        const int gg = lane >> 2, tq = lane & 3;
        if (tq < B) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int rl = warp * 16 + gg + 8 * half;
                const int R = r * ro + rl;
                const float s = half ? (c0[2] + c0[3] + c1[2] + c1[3]) : (c0[0] + c0[1] + c1[0] + c1[1]);
                long long f = fix_of(osc[rl] * s);
                if (h == 0) f += s_res[tq * ro + rl];
                red_add_fix(a.xa + (size_t)tq * H + R, f);
            }
        }
    }
    if (appender)
        #pragma unroll 1
        for (int i = tid; i < B * HD; i += kThreads) {
            const int b = i / HD, d = i - b * HD;
            const size_t slot = (((size_t)s_seq[b] * a.nkv + g) * a.cap + s_pos[b]) * HD + d;
            a.kc[slot] = __float2bfloat16_rn(kn[i]);
            a.vc[slot] = __float2bfloat16_rn(vn[i]);
        }
    if (bad && tid == 0) {
        set_status(a.status, kStatusTimeout);
        // let every copy this CTA started land before its shared memory goes away
        wait_phase(&bars[0], 0);
        wait_phase(&bars[1], 0);
        #pragma unroll 1
        for (int s = 0; s < S; ++s)
            if (s_last[s] >= 0) wait_phase(&bars[2 + s], (uint32_t)(s_last[s] / S) & 1u);
    }
    cluster_wait();  // no CTA leaves while a peer may still read its shared memory
}

// ===================================================================== FFN block
// CTA j (no cluster) serves FFN units [32 j, 32 j + 32): their 4 gate/up
// tiles (8 gate rows and the same 8 up units each, K = H whole) and k-pair j
// (the same 32 units) of every down row.
//  1. The RMSNorm-ed residual row (1 / rms and the gain in the operand) times
//     the 64 gate/up rows; warp w takes k-pairs [w KP / 8, (w + 1) KP / 8) of
//     all 4 tiles and the 8 warps' partial rows are summed in warp order.
//  2. a = silu(gate) * up for the 32 units, as the down operand.
//  3. Every down row times a (one k-pair per row tile, warp w taking tiles w,
//     w + 8, ...); the rows are added to the fixed-point residual stream, CTA
//     j also adding the stream's input to rows R = j (mod grid).
// With no exchange between CTAs there is no cluster barrier on the path; the
// price is H x B residual additions per CTA instead of H / 8 x B.
__global__ void __launch_bounds__(kThreads, 2) ffn_block_kernel(const FfnBlockArgs a) {
    constexpr int T = 2 * kFfnUnits / 16;  // gate/up tiles of the CTA
    static_assert(kStepMaxBatch * kFfnResidRows <= kThreads, "one residual input per thread");
    extern __shared__ __align__(128) unsigned char smem[];
    const FfnLayout L = ffn_layout(a.H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = blockIdx.x, G = gridDim.x;
    const int H = a.H, B = a.B, KP = H / 32, kpw = KP / kWarps, dtiles = H / 16;
    const uint32_t blob = (uint32_t)tile_blob_bytes(H), dblob = (uint32_t)tile_blob_bytes(a.I);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);  // 0 gate/up tiles, 1 down k-pairs
    float* s_sgu = reinterpret_cast<float*>(smem + L.sgu);
    float* s_sd = reinterpret_cast<float*>(smem + L.sd);
    float* s_red = reinterpret_cast<float*>(smem + L.red);
    long long* s_res = reinterpret_cast<long long*>(smem + L.resid);
    uint4* xop = reinterpret_cast<uint4*>(smem + L.xop);
    float* part = reinterpret_cast<float*>(smem + L.xop);  // [warp][sequence][64 rows], after the MMAs
    uint4* dop = reinterpret_cast<uint4*>(smem + L.dop);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bars[0], (uint32_t)T * blob);
        bulk_g2s(smem + L.wgu, a.wgu + (size_t)T * j * blob, (uint32_t)T * blob, &bars[0]);
        mbar_arrive_expect_tx(&bars[1], (uint32_t)dtiles * 512);
    }
    __syncthreads();
    if (warp == 0)
#pragma unroll 1
        for (int i = lane; i < dtiles; i += 32)
            bulk_g2s(smem + L.wd + (size_t)i * 512, a.wd + (size_t)i * dblob + kTileHeader + (size_t)j * 512, 512,
                     &bars[1]);
#pragma unroll 1
    for (int i = tid; i < 2 * kFfnUnits; i += kThreads) s_sgu[i] = a.gu_scale[(size_t)2 * kFfnUnits * j + i];
#pragma unroll 1
    for (int i = tid; i < H; i += kThreads) s_sd[i] = a.d_scale[i];
    pdl_wait();
    pdl_launch_dependents();

    // the stream's input at this CTA's rows R = j + i G (at most one per
    // thread: B nres <= 4 kFfnResidRows = kThreads), loaded now and parked in
    // shared memory after the gate/up rows
    const int nres = j < H ? (H - 1 - j) / G + 1 : 0;
    long long res_in = 0;
    if (tid < B * nres) res_in = __ldcg(a.xa + (size_t)(tid / nres) * H + j + (size_t)(tid % nres) * G);

    // ---- 1. gate/up rows times the normalised row, K split over the warps
    norm_operand(xop, a.xa, nullptr, nullptr, nullptr, B, H, a.ffn_norm, a.eps, s_red);
    bool bad = block_wait_failed(&bars[0], 0);
    float c0[T][4], c1[T][4];
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) c0[t][e] = c1[t][e] = 0.f;
    if (!bad)
#pragma unroll 1
        for (int p = warp * kpw; p < (warp + 1) * kpw; ++p) {
            const uint4 bv = xop[p * 32 + lane];
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const uint4 wv = *reinterpret_cast<const uint4*>(smem + L.wgu + (size_t)t * blob + kTileHeader +
                                                                 (size_t)p * 512 + lane * 16);
                mma_pair(c0[t], c1[t], wv, bv);
            }
        }
    if (tid < B * nres) s_res[(tid / nres) * kFfnResidRows + tid % nres] = res_in;
    __syncthreads();  // every warp is done with the operand: its space takes the partial rows
    {
        const int g = lane >> 2, q = lane & 3;
        float* pw = part + (warp * kStepMaxBatch + q) * (2 * kFfnUnits);
#pragma unroll
        for (int t = 0; t < T; ++t) {
            pw[t * 16 + g] = c0[t][0] + c0[t][1] + c1[t][0] + c1[t][1];
            pw[t * 16 + g + 8] = c0[t][2] + c0[t][3] + c1[t][2] + c1[t][3];
        }
    }
    __syncthreads();

    // ---- 2. a = silu(gate) * up for the CTA's units, as the down operand
    if (tid < B * kFfnUnits) {
        const int b = tid / kFfnUnits, u = tid - b * kFfnUnits;
        const int gr = (u >> 3) * 16 + (u & 7);  // gate row of unit u; its up row is gr + 8
        float sg = 0.f, su = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            sg += part[(w * kStepMaxBatch + b) * (2 * kFfnUnits) + gr];
            su += part[(w * kStepMaxBatch + b) * (2 * kFfnUnits) + gr + 8];
        }
        const float gate = s_sgu[gr] * sg, up = s_sgu[gr + 8] * su;
        const float v = (gate / (1.0f + expf(-gate))) * up;
        __half hi, lo;
        split_f16(v, hi, lo);
        __half* doph = reinterpret_cast<__half*>(dop);
        doph[frag_half(2 * b, u)] = hi;
        doph[frag_half(2 * b + 1, u)] = lo;
    }
    __syncthreads();

    // ---- 3. every down row over the CTA's units
    bad = block_wait_failed(&bars[1], 0) || bad;
    if (!bad) {
        const uint4 bv = dop[lane];
        const int g = lane >> 2, q = lane & 3;
#pragma unroll 1
        for (int t = warp; t < dtiles; t += kWarps) {
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_pair(d0, d1, *reinterpret_cast<const uint4*>(smem + L.wd + (size_t)t * 512 + lane * 16), bv);
            if (q < B) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int R = t * 16 + g + 8 * half;
                    const float s = half ? (d0[2] + d0[3] + d1[2] + d1[3]) : (d0[0] + d0[1] + d1[0] + d1[1]);
                    long long f = fix_of(s_sd[R] * s);
                    if (R % G == j) f += s_res[q * kFfnResidRows + R / G];
                    red_add_fix(a.xf + (size_t)q * H + R, f);
                }
            }
        }
    }
    if (bad && tid == 0) {
        set_status(a.status, kStatusTimeout);
        // let every copy this CTA started land before its shared memory goes away
        wait_phase(&bars[0], 0);
        wait_phase(&bars[1], 0);
    }
}

// ===================================================================== lm_head
// The tied embedding table swept once: a producer warp streams the CTA's
// range of 16-row tiles into a ring of S <= 8 shared-memory stages (the
// first stages before the wait), and consumer warp s takes the tiles of
// stage s (tile j -> stage and warp j % S) against the final-RMSNorm operand.  Each lane
// keeps the best (value, lowest index) key of its sequence; block, then
// grid atomicMax; the last CTA publishes the tokens.
__global__ void __launch_bounds__(kLmThreads, 2) lm_head_kernel(const LmHeadArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const LmLayout L = lm_layout(a.H, a.stages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.stages, H = a.H, B = a.B;
    const int ntiles = a.rows / 16;
    const int j0 = (int)((long long)ntiles * blockIdx.x / gridDim.x);
    const int n = (int)((long long)ntiles * (blockIdx.x + 1) / gridDim.x) - j0;
    const uint32_t blob = (uint32_t)tile_blob_bytes(H);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + S;
    unsigned long long* wbest = reinterpret_cast<unsigned long long*>(smem + L.best);
    float* s_inv = reinterpret_cast<float*>(smem + L.misc);
    float* s_red = s_inv + 4;
    int* s_abort = reinterpret_cast<int*>(s_red + 32);  // s_red: [8][4] sums of squares
    int* s_last = s_abort + 1;
    uint4* xop = reinterpret_cast<uint4*>(smem + L.xop);
    const bool producer = warp == kWarps && lane == 0;
    if (tid == 0) {
        #pragma unroll 1
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], 1);
        fence_mbar_init();
        *s_abort = 0;
        *s_last = 0;
    }
    __syncthreads();
    int issued = 0;
    auto issue = [&](int j) {
        const int s = j % S;
        mbar_arrive_expect_tx(&full[s], blob);
        bulk_g2s(smem + L.ring + (size_t)s * blob, a.w + (size_t)(j0 + j) * blob, blob, &full[s]);
    };
    if (producer)
        #pragma unroll 1
        for (; issued < S && issued < n; ++issued) issue(issued);
    float* s_gain = reinterpret_cast<float*>(smem + L.gain);
    #pragma unroll 1
    for (int i = tid; i < H; i += kLmThreads) s_gain[i] = a.final_norm[i];
    pdl_wait();
    pdl_launch_dependents();
    clear_share(a.clear, B * H);
    norm_operand(xop, a.xf, nullptr, nullptr, nullptr, B, H, s_gain, a.eps, s_red);

    if (producer) {
        #pragma unroll 1
        for (; issued < n; ++issued) {
            const int s = issued % S;
            if (*reinterpret_cast<volatile int*>(s_abort) ||
                !wait_phase(&empty[s], (uint32_t)(issued / S - 1) & 1u)) {
                *reinterpret_cast<volatile int*>(s_abort) = 1;
                break;
            }
            issue(issued);
        }
        *s_last = issued;
    }
    unsigned long long best = 0ull;
    if (warp < kWarps) {
        const int kpairs = H / 32;
        const int gg = lane >> 2, tq = lane & 3;
        // stage s belongs to consumer warp s alone (tile j -> stage and warp j % S), so every wait on a
        // stage's full barrier is for the phase right after the one that warp last consumed
        for (int j = warp; warp < S && j < n; j += S) {
            const int s = j % S;
            if (*reinterpret_cast<volatile int*>(s_abort)) break;
            if (!wait_phase(&full[s], (uint32_t)(j / S) & 1u)) {
                *reinterpret_cast<volatile int*>(s_abort) = 1;
                break;
            }
            const unsigned char* wt = smem + L.ring + (size_t)s * blob;
            float c[4][4];
#pragma unroll
            for (int x = 0; x < 4; ++x) c[x][0] = c[x][1] = c[x][2] = c[x][3] = 0.f;
            for (int p = 0; p < kpairs; p += 2) {
                const uint4 w0 = *reinterpret_cast<const uint4*>(wt + kTileHeader + (size_t)p * 512 + lane * 16);
                const uint4 w1 = *reinterpret_cast<const uint4*>(wt + kTileHeader + (size_t)(p + 1) * 512 + lane * 16);
                mma_pair(c[0], c[1], w0, xop[p * 32 + lane]);
                mma_pair(c[2], c[3], w1, xop[(p + 1) * 32 + lane]);
            }
            const float* sc = reinterpret_cast<const float*>(wt);
            const float sc0 = sc[gg], sc1 = sc[gg + 8];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const float v0 = sc0 * (c[0][0] + c[0][1] + c[1][0] + c[1][1] + c[2][0] + c[2][1] + c[3][0] + c[3][1]);
            const float v1 = sc1 * (c[0][2] + c[0][3] + c[1][2] + c[1][3] + c[2][2] + c[2][3] + c[3][2] + c[3][3]);
            const int row0 = (j0 + j) * 16 + gg, row1 = row0 + 8;
            if (tq < B) {
                if (row0 < a.valid_rows) {
                    if (a.logits) a.logits[(size_t)tq * a.valid_rows + row0] = v0;
                    const unsigned long long k0 = argmax_key(v0, (uint32_t)row0);
                    best = k0 > best ? k0 : best;
                }
                if (row1 < a.valid_rows) {
                    if (a.logits) a.logits[(size_t)tq * a.valid_rows + row1] = v1;
                    const unsigned long long k1 = argmax_key(v1, (uint32_t)row1);
                    best = k1 > best ? k1 : best;
                }
            }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
        if (lane < 4) wbest[warp * 4 + lane] = best;
    }
    __syncthreads();
    __shared__ int is_last;
    if (tid < B) {
        unsigned long long k = 0ull;
        for (int w = 0; w < kWarps; ++w) k = wbest[w * 4 + tid] > k ? wbest[w * 4 + tid] : k;
        atomicMax(&a.keys[tid], k);
    }
    if (*reinterpret_cast<volatile int*>(s_abort) && tid == 0) {
        set_status(a.status, kStatusTimeout);
        #pragma unroll 1
        for (int s = 0; s < S; ++s) {
            // the last tile issued into stage s, if any
            const int last = *s_last - 1 - ((*s_last - 1 - s) % S + S) % S;
            if (last >= 0 && last < *s_last) wait_phase(&full[s], (uint32_t)(last / S) & 1u);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
    __syncthreads();
    if (is_last) {
        __threadfence();
        const int step = *reinterpret_cast<volatile int32_t*>(a.step);
        if (tid < B) {
            const unsigned long long k = atomicExch(&a.keys[tid], 0ull);
            const int tok = (int)argmax_key_index(k);
            a.tokens[tid] = tok;
            if (step < a.out_cap) a.out_ids[(size_t)tid * a.out_cap + step] = tok;
            if (a.advance_pos) a.pos[tid] += 1;
        }
        __syncthreads();
        if (tid == 0) {
            *a.step = step + 1;
            *a.counter = 0u;
        }
    }
}

// ===================================================================== host side
size_t attn_block_smem(int H, int hd, int kv_stages) { return attn_block_layout(H, hd, kv_stages).total; }
size_t ffn_block_smem(int H) { return ffn_layout(H).total; }
size_t lm_head_smem(int H, int stages) { return lm_layout(H, stages).total; }

bool step_plan(const StepShape& s, int num_sms, int smem_optin, StepPlan* p) {
    if (s.hd != 64 && s.hd != 128) return false;
    if (s.nkv < 1 || s.nh % s.nkv) return false;
    // K slices of whole k-pairs, at most 4 per CTA (a sequence's operand threads share one warp)
    if (s.H % 256 || s.H > 1024 || s.I % kFfnUnits || s.vocab_rows % 16) return false;
    if ((s.H + s.I / kFfnUnits - 1) / (s.I / kFfnUnits) > kFfnResidRows) return false;  // input rows per FFN CTA
    StepPlan q;
    q.kv_stages = p->kv_stages < 1 ? 2 : p->kv_stages;
    if (attn_block_smem(s.H, s.hd, q.kv_stages) > (size_t)smem_optin) return false;
    if (ffn_block_smem(s.H) > (size_t)smem_optin) return false;
    q.ffn_grid = s.I / kFfnUnits;
    q.lm_stages = 6;
    while (q.lm_stages > 2 && lm_head_smem(s.H, q.lm_stages) > (size_t)smem_optin) --q.lm_stages;
    if (lm_head_smem(s.H, q.lm_stages) > (size_t)smem_optin) return false;
    q.lm_grid = std::min(num_sms, s.vocab_rows / 16);
    *p = q;
    return true;
}

bool step_prepare_device() {
    const void* fns[] = {(const void*)attn_block_kernel<64>, (const void*)attn_block_kernel<128>,
                         (const void*)ffn_block_kernel, (const void*)lm_head_kernel};
    for (const void* f : fns)
        if (allow_max_dynamic_smem(f) != cudaSuccess) return false;
    return true;
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_ex(void (*kern)(KArgs...), int grid, int block, size_t smem, int cluster, cudaStream_t st,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    int na = 0;
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster > 1) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = cluster;
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = at;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_attn_block(const AttnBlockArgs& a, int hd, cudaStream_t st) {
    const size_t smem = attn_block_smem(a.H, hd, a.kv_stages);
    const int grid = a.nh * kClusterCtas;
    if (hd == 128) return launch_ex(attn_block_kernel<128>, grid, kThreads, smem, kClusterCtas, st, a);
    if (hd == 64) return launch_ex(attn_block_kernel<64>, grid, kThreads, smem, kClusterCtas, st, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_ffn_block(const FfnBlockArgs& a, int grid, cudaStream_t st) {
    return launch_ex(ffn_block_kernel, grid, kThreads, ffn_block_smem(a.H), 1, st, a);
}

cudaError_t launch_lm_head(const LmHeadArgs& a, int grid, cudaStream_t st) {
    return launch_ex(lm_head_kernel, grid, kLmThreads, lm_head_smem(a.H, a.stages), 1, st, a);
}

static int max_clusters(const void* f, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterCtas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kClusterCtas;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int attn_block_max_clusters(int H, int hd, int kv_stages) {
    const void* f = hd == 128 ? (const void*)attn_block_kernel<128> : (const void*)attn_block_kernel<64>;
    return max_clusters(f, attn_block_smem(H, hd, kv_stages));
}

int ffn_block_max_blocks(int H) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ffn_block_kernel, kThreads, ffn_block_smem(H)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace q3
