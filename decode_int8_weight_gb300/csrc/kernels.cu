// q3i8 kernels: decode step pieces and the plain prefill pieces (sm_103a).
//
// The decoder block computed here is the Qwen3 family's ("Model-agnostic LLM
// inference", section "Supported models"): RMSNorm -> QKV -> per-head
// RMSNorm on Q and K -> RoPE -> KV append (bf16) -> grouped-query attention
// -> O + residual -> RMSNorm -> SiLU-gated FFN + residual, then a final
// RMSNorm and the tied lm_head with a fused argmax ("Run local LLM decode",
// section "Limitations": every token is the argmax at its step).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

size_t packed_offset(int row, int k, int K) {
    int tile = row >> 4, r = row & 15, g = r & 7, hi_row = r >> 3;
    int pair = k >> 5, kin = k & 31, kstep = kin >> 4, kk = kin & 15;
    int t = (kk & 7) >> 1, hi_k = kk >> 3, sub = kk & 1;
    int lane = 4 * g + t;
    int byte = 4 * hi_k + 2 * hi_row + sub;
    return (size_t)tile * (kTileHeader + 16 * (size_t)K) + kTileHeader + (size_t)pair * 512 + lane * 16 + kstep * 8 +
           byte;
}

// =====================================================================
// int8 weight GEMV / skinny GEMM on the tensor cores.
//
// y[b][row] = scale[row] * sum_k q[row][k] * x[b][k] for B <= 4*NT rows of
// activations.  Each warp takes every 8th pair of k-steps of a 16-row
// weight tile (split-K inside the CTA); one 16-byte streaming load per lane
// carries the tile's bytes for two m16n8k16 MMAs, converted to f16 in
// registers (exact for |q| <= 127).  The activation operand holds each
// sequence as two f16 columns (hi and lo parts of the fp32 value), so one
// weight tile serves all B sequences and the fp32 value is kept to ~22 bits.
// The 8 warps' partial sums meet in shared memory; the epilogue applies the
// row scale and the mode's fusion.
// =====================================================================
// Work items of one CTA whose weights it asks L2 for ahead of use: the
// first ones before waiting on the previous kernel, then each item's
// successor this far ahead.
constexpr int kGemvPrefetchItems = 2;
constexpr bool kGemvRollingPrefetch = true;

// Ask L2 for the weight bytes of work item `item` (4 KB requests spread over
// the CTA's threads).
Q3_DEV void gemv_prefetch_item(const GemvArgs& a, int item, int ks, int kpairs) {
    const int tile = item / ks, part = item - tile * ks;
    const int p_lo = (int)((long long)kpairs * part / ks), p_hi = (int)((long long)kpairs * (part + 1) / ks);
    const uint8_t* base = a.w + (size_t)tile * (kTileHeader + 16 * (size_t)a.K) + kTileHeader + (size_t)p_lo * 512;
    const uint32_t bytes = (uint32_t)(p_hi - p_lo) * 512u;
    for (uint32_t off = threadIdx.x * 4096u; off < bytes; off += blockDim.x * 4096u)
        prefetch_l2_bulk(base + off, bytes - off < 4096u ? bytes - off : 4096u);
}

// Fixed-point sums of squares (value * 2^32) of the folded RMSNorm.
Q3_DEV long long ss_fix(float v) { return __float2ll_rn(v * 0x1p32f); }
Q3_DEV float ss_float(long long x) { return __ll2float_rn(x) * 0x1p-32f; }

template <int NT, int MODE>
__global__ void __launch_bounds__(256) gemv_kernel(GemvArgs a) {
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int n_tiles = a.rows >> 4;
    const int kpairs = a.K >> 5;
    const int ks = (MODE == kResid && a.ksplit > 1) ? a.ksplit : 1;
    // The weights do not depend on the previous kernel: start moving this
    // CTA's first items into L2 while that kernel finishes.
    for (int j = 0; j < kGemvPrefetchItems; ++j) {
        const int item = blockIdx.x + j * gridDim.x;
        if (item >= n_tiles * ks) break;
        gemv_prefetch_item(a, item, ks, kpairs);
    }
    pdl_wait();
    __shared__ float red[8][NT][32][2];
    __shared__ unsigned long long best[4 * NT];
    __shared__ int is_last;
    __shared__ float s_inv[4 * NT];   // folded RMSNorm: 1 / rms per sequence (1 without)
    __shared__ float s_sq[NT * 64];   // folded RMSNorm: x^2 of the tile's rows
    if (a.ss_clear && blockIdx.x == 0)
        for (int b = threadIdx.x; b < a.B; b += blockDim.x) a.ss_clear[b] = 0;
    for (int b = threadIdx.x; b < 4 * NT; b += blockDim.x)
        s_inv[b] = (a.ss_in && b < a.B) ? 1.0f / sqrtf(ss_float(__ldcg(a.ss_in + b)) / (float)a.norm_H + a.eps) : 1.0f;
    __syncthreads();

    if (MODE == kArgmax) {
        for (int i = threadIdx.x; i < 4 * NT; i += blockDim.x) best[i] = 0ull;
        __syncthreads();
    }
    // work item = (tile, K part); residual tiles may be split over ks CTAs
    for (int item = blockIdx.x; item < n_tiles * ks; item += gridDim.x) {
        if (kGemvRollingPrefetch) {
            const long long ahead = item + (long long)kGemvPrefetchItems * gridDim.x;
            if (ahead < (long long)n_tiles * ks) gemv_prefetch_item(a, (int)ahead, ks, kpairs);
        }
        const int tile = item / ks, part = item - tile * ks;
        const int p_lo = (int)((long long)kpairs * part / ks), p_hi = (int)((long long)kpairs * (part + 1) / ks);
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        const uint8_t* wt = a.w + (size_t)tile * (kTileHeader + 16 * (size_t)a.K) + kTileHeader + lane * 16;
#pragma unroll 4
        for (int p = p_lo + warp; p < p_hi; p += 8) {
            uint4 wv = ld_stream_u4(wt + (size_t)p * 512);
            uint32_t A0[4], A1[4];
            u8x4_to_f16x2x2(wv.x, A0[0], A0[1]);
            u8x4_to_f16x2x2(wv.y, A0[2], A0[3]);
            u8x4_to_f16x2x2(wv.z, A1[0], A1[1]);
            u8x4_to_f16x2x2(wv.w, A1[2], A1[3]);
            const int k0 = p * 32 + 2 * t;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                uint32_t b0, b1, b2, b3;
                if (a.xfrag) {
                    const uint4 bw = *reinterpret_cast<const uint4*>(a.xh + ((((size_t)p * 8 + n) * 32 + lane) << 3));
                    b0 = bw.x, b1 = bw.y, b2 = bw.z, b3 = bw.w;
                } else {
                    const __half* xr = a.xh + (size_t)(8 * n + g) * a.K + k0;
                    b0 = *reinterpret_cast<const uint32_t*>(xr);
                    b1 = *reinterpret_cast<const uint32_t*>(xr + 8);
                    b2 = *reinterpret_cast<const uint32_t*>(xr + 16);
                    b3 = *reinterpret_cast<const uint32_t*>(xr + 24);
                }
                mma_f16_16816(acc[n], A0, b0, b1);
                mma_f16_16816(acc[n], A1, b2, b3);
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            red[warp][n][lane][0] = acc[n][0] + acc[n][1];  // row g,   sequence 4n+t (hi + lo)
            red[warp][n][lane][1] = acc[n][2] + acc[n][3];  // row g+8, sequence 4n+t
        }
        __syncthreads();
        if (MODE == kSiluGate) {
            // tile rows 0..7 are gate rows, 8..15 the up rows of the same 8 units
            for (int i = threadIdx.x; i < NT * 32; i += blockDim.x) {
                const int n = i >> 5, ln = i & 31, gg = ln >> 2, b = 4 * n + (ln & 3);
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    s0 += red[w][n][ln][0];
                    s1 += red[w][n][ln][1];
                }
                if (b < a.B) {
                    const int rg = tile * 16 + gg;
                    const float gate = a.scale[rg] * s0 * s_inv[b];
                    const float up = a.scale[rg + 8] * s1 * s_inv[b];
                    const float v = (gate / (1.0f + expf(-gate))) * up;
                    const int idx = tile * 8 + gg;
                    __half hi, lo;
                    split_f16(v, hi, lo);
                    a.yh[plane_index(2 * b, idx, a.ldyh, a.yfrag)] = hi;
                    a.yh[plane_index(2 * b + 1, idx, a.ldyh, a.yfrag)] = lo;
                }
            }
        } else if (MODE == kResid && ks > 1 && a.kpart) {
            // split K: park this part's sums; the tile's last part to finish adds
            // all parts in order, so the result does not depend on timing
            float* kp = a.kpart + ((size_t)tile * ks + part) * (NT * 64);
            for (int i = threadIdx.x; i < NT * 64; i += blockDim.x) {
                const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) sum += red[w][n][ln][half];
                kp[i] = sum;
            }
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) is_last = (atomicAdd(a.tile_cnt + tile, 1u) == (unsigned)(ks - 1));
            __syncthreads();
            if (is_last) {
                __threadfence();
                for (int i = threadIdx.x; i < NT * 64; i += blockDim.x) {
                    const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, gg = ln >> 2, b = 4 * n + (ln & 3);
                    float sum = 0.f;
                    for (int q = 0; q < ks; ++q) sum += __ldcg(a.kpart + ((size_t)tile * ks + q) * (NT * 64) + i);
                    float xs = 0.f;
                    if (b < a.B) {
                        const int row = tile * 16 + gg + 8 * half;
                        float* p = a.y + (size_t)b * a.ldy + row;
                        xs = *p + a.scale[row] * sum;
                        *p = xs;
                        if (a.norm_g) {
                            __half hi, lo;
                            split_f16(__fmul_rn(xs, a.norm_g[row]), hi, lo);
                            a.norm_xh[plane_index(2 * b, row, a.norm_H, 1)] = hi;
                            a.norm_xh[plane_index(2 * b + 1, row, a.norm_H, 1)] = lo;
                        }
                    }
                    s_sq[i] = xs * xs;
                }
                if (a.norm_g) {
                    // sequence b's 16 rows of this tile, in a fixed order
                    __syncthreads();
                    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
                        const int n = b >> 2, t = b & 3;
                        float sq = 0.f;
                        for (int gg = 0; gg < 8; ++gg)
                            sq += s_sq[n * 64 + (4 * gg + t) * 2] + s_sq[n * 64 + (4 * gg + t) * 2 + 1];
                        atomicAdd(reinterpret_cast<unsigned long long*>(a.ss_out + b), (unsigned long long)ss_fix(sq));
                    }
                }
                if (threadIdx.x == 0) a.tile_cnt[tile] = 0u;
            }
        } else {
            for (int i = threadIdx.x; i < NT * 64; i += blockDim.x) {
                const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, gg = ln >> 2, b = 4 * n + (ln & 3);
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) sum += red[w][n][ln][half];
                if (b < a.B) {
                    const int row = tile * 16 + gg + 8 * half;
                    const float v = a.scale[row] * sum * s_inv[b];
                    if (MODE == kStore) {
                        a.y[(size_t)b * a.ldy + row] = v;
                    } else if (MODE == kResid) {
                        float* p = a.y + (size_t)b * a.ldy + row;
                        if (ks > 1) atomicAdd(p, v);  // split K without kpart: parts meet in atomic adds
                        else *p = *p + v;
                    } else {
                        if (row < a.valid_rows) {
                            if (a.logits) a.logits[(size_t)b * a.valid_rows + row] = v;
                            atomicMax(&best[b], argmax_key(v, (uint32_t)row));
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
    if (MODE == kArgmax) {
        // block result -> grid result; the last block to finish publishes the tokens
        if (threadIdx.x < a.B) atomicMax(&a.keys[threadIdx.x], best[threadIdx.x]);
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) is_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
        __syncthreads();
        if (is_last) {
            __threadfence();
            const int step = *reinterpret_cast<volatile int32_t*>(a.step);
            if (threadIdx.x < a.B) {
                const int b = threadIdx.x;
                const unsigned long long k = atomicExch(&a.keys[b], 0ull);
                const int tok = (int)argmax_key_index(k);
                a.tokens[b] = tok;
                if (step < a.out_cap) a.out_ids[(size_t)b * a.out_cap + step] = tok;
                if (a.advance_pos) a.pos[b] += 1;
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                *a.step = step + 1;
                *a.counter = 0u;
            }
        }
    }
}

// =====================================================================
// The same GEMV with the CTA's weights staged before the wait.
//
// One CTA per (tile, K part): its slice of the tile blob is one contiguous
// run of k-pairs, which thread 0 bulk-copies into shared memory, and the
// tile's row scales (and, for the residual mode, the next norm's gains) are
// read, all before waiting on the previous kernel: that kernel's tail hides
// the weight fetch.  After the wait the CTA reads only what the previous
// kernels wrote (the operand planes, the sums of squares, the residual
// rows), issued before the MMAs.  When K is split (kResid), the ks CTAs of a
// tile form a thread-block cluster: each parks its part's sums in its shared
// memory and CTA 0 of the cluster adds the parts in order through
// distributed shared memory, so the result has the same bits as the parked
// parts of gemv_kernel and needs no counter or second pass through global
// memory.  Used by the decode step (fragment-ordered operand planes) and by
// the prefill of up to 32 rows per chunk (plain planes); the epilogues are
// gemv_kernel's.
// =====================================================================
constexpr uint32_t kGemvStageMax = 64u * 1024u;  // largest weight slice staged (bytes)

template <int NT, int MODE, bool FRAG>
__global__ void __launch_bounds__(256, NT >= 8 ? (MODE == kSiluGate ? 3 : 2) : (NT == 1 && MODE == kSiluGate ? 6 : 1))
gemv_staged_kernel(GemvArgs a) {
    if (!a.late_dependents) pdl_launch_dependents();
    extern __shared__ __align__(128) unsigned char wsm[];
    __shared__ float red[8][NT][32][2];
    __shared__ float s_part[NT * 64];  // this CTA's sums (the tile's, or its K part's)
    __shared__ float s_sq[NT * 64];
    __shared__ float s_inv[4 * NT];
    __shared__ float s_scale[16], s_gain[16];
    __shared__ __align__(8) uint64_t wbar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = (MODE == kResid && a.ksplit > 1) ? a.ksplit : 1;
    const int tile = blockIdx.x / ks, part = blockIdx.x - tile * ks;
    const int kpairs = a.K >> 5;
    const int p_lo = (int)((long long)kpairs * part / ks), p_hi = (int)((long long)kpairs * (part + 1) / ks);
    const bool lead = part == 0;  // cluster rank 0 (ks > 1) adds the parts and writes the tile
    if (threadIdx.x == 0) {
        mbar_init(&wbar, 1);
        fence_mbar_init();
        const uint32_t bytes = (uint32_t)(p_hi - p_lo) * 512u;
        mbar_arrive_expect_tx(&wbar, bytes);
        bulk_g2s(wsm, a.w + (size_t)tile * (kTileHeader + 16 * (size_t)a.K) + kTileHeader + (size_t)p_lo * 512, bytes,
                 &wbar);
    }
    if (threadIdx.x < 16) {
        s_scale[threadIdx.x] = a.scale[tile * 16 + threadIdx.x];
        s_gain[threadIdx.x] = (MODE == kResid && a.norm_g) ? a.norm_g[tile * 16 + threadIdx.x] : 0.f;
    }
    __syncthreads();  // the barrier is initialised before anyone waits on it
    pdl_wait();
    if (a.late_dependents) pdl_launch_dependents();

    // reads of what earlier kernels wrote, in flight during the MMAs
    long long ss = 0;
    if (a.ss_in && threadIdx.x < a.B) ss = __ldcg(a.ss_in + threadIdx.x);
    constexpr int kEpi = (NT * 64 + 255) / 256;  // epilogue elements per thread
    float yin[kEpi];
#pragma unroll
    for (int j = 0; j < kEpi; ++j) {
        yin[j] = 0.f;
        const int i = threadIdx.x + 256 * j;
        if (MODE == kResid && lead && i < NT * 64) {
            const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, b = 4 * n + (ln & 3);
            if (b < a.B) yin[j] = a.y[(size_t)b * a.ldy + tile * 16 + (ln >> 2) + 8 * half];
        }
    }
    if (a.ss_clear && blockIdx.x == 0)
        for (int b = threadIdx.x; b < a.B; b += blockDim.x) a.ss_clear[b] = 0;

    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    const bool ok = mbar_wait_bounded(&wbar, 0);
    if (ok) {
        const uint32_t wbase = smem_u32(wsm) + lane * 16;
#pragma unroll(NT >= 4 ? 2 : 4)
        for (int p = p_lo + warp; p < p_hi; p += 8) {
            const uint4 wv = lds128(wbase + (uint32_t)(p - p_lo) * 512u);
            uint32_t A0[4], A1[4];
            u8x4_to_f16x2x2(wv.x, A0[0], A0[1]);
            u8x4_to_f16x2x2(wv.y, A0[2], A0[3]);
            u8x4_to_f16x2x2(wv.z, A1[0], A1[1]);
            u8x4_to_f16x2x2(wv.w, A1[2], A1[3]);
            // all tiles' first k-steps, then their second ones: no MMA waits on the one before it
            uint4 bw[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if constexpr (FRAG) {
                    bw[n] = *reinterpret_cast<const uint4*>(a.xh + ((((size_t)p * 8 + n) * 32 + lane) << 3));
                } else {
                    const __half* xr = a.xh + (size_t)(8 * n + (lane >> 2)) * a.K + p * 32 + 2 * (lane & 3);
                    bw[n].x = *reinterpret_cast<const uint32_t*>(xr);
                    bw[n].y = *reinterpret_cast<const uint32_t*>(xr + 8);
                    bw[n].z = *reinterpret_cast<const uint32_t*>(xr + 16);
                    bw[n].w = *reinterpret_cast<const uint32_t*>(xr + 24);
                }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) mma_f16_16816(acc[n], A0, bw[n].x, bw[n].y);
#pragma unroll
            for (int n = 0; n < NT; ++n) mma_f16_16816(acc[n], A1, bw[n].z, bw[n].w);
        }
    } else {
        set_status(a.status, kStatusTimeout);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        red[warp][n][lane][0] = acc[n][0] + acc[n][1];  // row g,   sequence 4n+t (hi + lo)
        red[warp][n][lane][1] = acc[n][2] + acc[n][3];  // row g+8, sequence 4n+t
    }
    if (threadIdx.x < 4 * NT)
        s_inv[threadIdx.x] = (a.ss_in && threadIdx.x < a.B)
                                 ? 1.0f / sqrtf(ss_float(ss) / (float)a.norm_H + a.eps)
                                 : 1.0f;
    __syncthreads();
    for (int i = threadIdx.x; i < NT * 64; i += blockDim.x) {
        const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sum += red[w][n][ln][half];
        s_part[i] = sum;
    }
    if (MODE == kResid && ks > 1) {
        cluster_arrive();
        cluster_wait();  // every part is visible in the cluster
        if (lead)
            for (int i = threadIdx.x; i < NT * 64; i += blockDim.x) {
                float sum = 0.f;
                for (int q = 0; q < ks; ++q) sum += peer(s_part, q)[i];
                s_sq[i] = sum;  // the tile's sums (s_sq is free until the epilogue below)
            }
        cluster_arrive();  // done with the peers' shared memory
        cluster_wait();    // no CTA leaves while the lead may still read it
        if (!lead) {
            if (!ok) mbar_wait_bounded(&wbar, 0);
            return;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < NT * 64; i += blockDim.x) s_part[i] = s_sq[i];
    }
    __syncthreads();

    if (MODE == kSiluGate) {
        // tile rows 0..7 are gate rows, 8..15 the up rows of the same 8 units
        for (int i = threadIdx.x; i < NT * 32; i += blockDim.x) {
            const int n = i >> 5, ln = i & 31, gg = ln >> 2, b = 4 * n + (ln & 3);
            if (b < a.B) {
                const float gate = s_scale[gg] * s_part[n * 64 + 2 * ln] * s_inv[b];
                const float up = s_scale[gg + 8] * s_part[n * 64 + 2 * ln + 1] * s_inv[b];
                const float v = (gate / (1.0f + expf(-gate))) * up;
                const int idx = tile * 8 + gg;
                __half hi, lo;
                split_f16(v, hi, lo);
                a.yh[plane_index(2 * b, idx, a.ldyh, a.yfrag)] = hi;
                a.yh[plane_index(2 * b + 1, idx, a.ldyh, a.yfrag)] = lo;
            }
        }
    } else if (MODE == kResid) {
#pragma unroll
        for (int j = 0; j < kEpi; ++j) {
            const int i = threadIdx.x + 256 * j;
            if (i >= NT * 64) break;
            const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, gg = ln >> 2, b = 4 * n + (ln & 3);
            float xs = 0.f;
            if (b < a.B) {
                const int r16 = gg + 8 * half, row = tile * 16 + r16;
                xs = yin[j] + s_scale[r16] * s_part[i];
                a.y[(size_t)b * a.ldy + row] = xs;
                if (a.norm_g) {
                    __half hi, lo;
                    split_f16(__fmul_rn(xs, s_gain[r16]), hi, lo);
                    a.norm_xh[plane_index(2 * b, row, a.norm_H, 1)] = hi;
                    a.norm_xh[plane_index(2 * b + 1, row, a.norm_H, 1)] = lo;
                }
            }
            s_sq[i] = xs * xs;
        }
        if (a.norm_g) {
            // sequence b's 16 rows of this tile, in a fixed order
            __syncthreads();
            for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
                const int n = b >> 2, t = b & 3;
                float sq = 0.f;
                for (int gg = 0; gg < 8; ++gg)
                    sq += s_sq[n * 64 + (4 * gg + t) * 2] + s_sq[n * 64 + (4 * gg + t) * 2 + 1];
                atomicAdd(reinterpret_cast<unsigned long long*>(a.ss_out + b), (unsigned long long)ss_fix(sq));
            }
        }
    } else {
        for (int i = threadIdx.x; i < NT * 64; i += blockDim.x) {
            const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, gg = ln >> 2, b = 4 * n + (ln & 3);
            if (b < a.B) {
                const int r16 = gg + 8 * half;
                a.y[(size_t)b * a.ldy + tile * 16 + r16] = s_scale[r16] * s_part[i] * s_inv[b];
            }
        }
    }
    if (!ok && threadIdx.x == 0) mbar_wait_bounded(&wbar, 0);
}

// =====================================================================
// The lm_head sweep with its argmax for B > 4 (several column tiles).
//
// gemv_kernel splits K over the warps of a CTA, so every weight tile makes
// each warp read its share of all NT activation tiles again from L2 (8x the
// weight bytes at NT = 8).  Here the activation planes (NT column tiles of
// every k-pair, fragment order) are bulk-copied into shared memory once per
// CTA, and each warp takes whole weight tiles (all of K) in turn: it streams
// a tile's bytes from global memory in batches of head_batch k-pairs (asking
// L2 for its next tile meanwhile) and keeps the running argmax key of each
// of its lanes' sequences in registers.  No partial sums cross warps.  The
// keys meet in shared memory, then in global memory; the last CTA publishes
// the tokens as gemv_kernel does.  The dot products are summed over K in
// k-pair order by one warp.
// =====================================================================
// k-pairs of weights per batch (two batches in flight per warp); 2 at 8
// column tiles, where 16 warps per SM share the latency
template <int NT>
__host__ __device__ constexpr int head_batch() { return NT >= 8 ? 2 : 4; }

Q3_DEV void prefetch_tile_l2(const uint8_t* tile_base, uint32_t bytes, int lane) {
    for (uint32_t off = (uint32_t)lane * 4096u; off < bytes; off += 32u * 4096u)
        prefetch_l2_bulk(tile_base + off, bytes - off < 4096u ? bytes - off : 4096u);
}

// Threads per CTA: at 8 column tiles one CTA fills an SM's shared memory, so
// it takes 16 warps to hide the MMA and conversion latencies.
template <int NT>
__host__ __device__ constexpr int head_threads() { return NT >= 8 ? 512 : 256; }

template <int NT>
__global__ void __launch_bounds__(head_threads<NT>()) lm_head_wide_kernel(GemvArgs a) {
    pdl_launch_dependents();
    extern __shared__ __align__(128) unsigned char xs[];  // [kpairs][NT][32 lanes][16 B]
    __shared__ __align__(8) uint64_t xbar;
    __shared__ unsigned long long best[4 * NT];
    __shared__ float s_inv[4 * NT];
    __shared__ int is_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int n_tiles = a.rows >> 4, kpairs = a.K >> 5;
    constexpr int kW = head_threads<NT>() / 32;  // warps per CTA
    constexpr int kHeadBatch = head_batch<NT>();
    const int nw = gridDim.x * kW;
    const size_t blob = kTileHeader + 16 * (size_t)a.K;
    const uint32_t wbytes = 16u * (uint32_t)a.K;
    int tile = blockIdx.x * kW + warp;
    // the weights do not depend on the previous kernel
    if (tile < n_tiles) prefetch_tile_l2(a.w + (size_t)tile * blob + kTileHeader, wbytes, lane);
    if (threadIdx.x == 0) {
        mbar_init(&xbar, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 4 * NT) best[threadIdx.x] = 0ull;
    __syncthreads();
    pdl_wait();
    if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(&xbar, (uint32_t)kpairs * NT * 512u);
        __syncwarp();
        for (int p = lane; p < kpairs; p += 32)
            bulk_g2s(xs + (size_t)p * NT * 512, reinterpret_cast<const uint8_t*>(a.xh) + (size_t)p * 8 * 512,
                     NT * 512u, &xbar);
    }
    if (a.ss_clear && blockIdx.x == 0)
        for (int b = threadIdx.x; b < a.B; b += blockDim.x) a.ss_clear[b] = 0;
    if (threadIdx.x < 4 * NT)
        s_inv[threadIdx.x] = (a.ss_in && threadIdx.x < a.B)
                                 ? 1.0f / sqrtf(ss_float(__ldcg(a.ss_in + threadIdx.x)) / (float)a.norm_H + a.eps)
                                 : 1.0f;
    __syncthreads();
    const bool ok = mbar_wait_bounded(&xbar, 0);
    if (!ok) set_status(a.status, kStatusTimeout);

    unsigned long long kb[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) kb[n] = 0ull;
    const uint32_t xbase = smem_u32(xs) + lane * 16;
    for (; ok && tile < n_tiles; tile += nw) {
        if (tile + nw < n_tiles) prefetch_tile_l2(a.w + (size_t)(tile + nw) * blob + kTileHeader, wbytes, lane);
        const int r0 = tile * 16 + g, r1 = r0 + 8;
        const float sc0 = a.scale[r0], sc1 = a.scale[r1];
        const uint8_t* wt = a.w + (size_t)tile * blob + kTileHeader + lane * 16;
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        uint4 wv[kHeadBatch], wn[kHeadBatch];
#pragma unroll
        for (int u = 0; u < kHeadBatch; ++u)
            if (u < kpairs) wv[u] = ld_stream_u4(wt + (size_t)u * 512);
        for (int p0 = 0; p0 < kpairs; p0 += kHeadBatch) {
            // the next batch is in flight while this one is multiplied
#pragma unroll
            for (int u = 0; u < kHeadBatch; ++u)
                if (p0 + kHeadBatch + u < kpairs) wn[u] = ld_stream_u4(wt + (size_t)(p0 + kHeadBatch + u) * 512);
#pragma unroll
            for (int u = 0; u < kHeadBatch; ++u) {
                if (p0 + u >= kpairs) break;
                uint32_t A0[4], A1[4];
                u8x4_to_f16x2x2(wv[u].x, A0[0], A0[1]);
                u8x4_to_f16x2x2(wv[u].y, A0[2], A0[3]);
                u8x4_to_f16x2x2(wv[u].z, A1[0], A1[1]);
                u8x4_to_f16x2x2(wv[u].w, A1[2], A1[3]);
                // all tiles' first k-steps, then their second ones
                uint4 bw[NT];
#pragma unroll
                for (int n = 0; n < NT; ++n) bw[n] = lds128(xbase + (uint32_t)((p0 + u) * NT + n) * 512u);
#pragma unroll
                for (int n = 0; n < NT; ++n) mma_f16_16816(acc[n], A0, bw[n].x, bw[n].y);
#pragma unroll
                for (int n = 0; n < NT; ++n) mma_f16_16816(acc[n], A1, bw[n].z, bw[n].w);
            }
#pragma unroll
            for (int u = 0; u < kHeadBatch; ++u) wv[u] = wn[u];
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int b = 4 * n + t;
            if (b >= a.B) continue;
            const float v0 = sc0 * (acc[n][0] + acc[n][1]) * s_inv[b];  // row r0, sequence b (hi + lo)
            const float v1 = sc1 * (acc[n][2] + acc[n][3]) * s_inv[b];  // row r1
            if (r0 < a.valid_rows) {
                if (a.logits) a.logits[(size_t)b * a.valid_rows + r0] = v0;
                kb[n] = max(kb[n], argmax_key(v0, (uint32_t)r0));
            }
            if (r1 < a.valid_rows) {
                if (a.logits) a.logits[(size_t)b * a.valid_rows + r1] = v1;
                kb[n] = max(kb[n], argmax_key(v1, (uint32_t)r1));
            }
        }
    }
    // lanes t, t + 4, ... hold the same sequences: their maximum, then the CTA's
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) kb[n] = max(kb[n], __shfl_xor_sync(0xffffffffu, kb[n], o));
        if (g == 0 && 4 * n + t < a.B) atomicMax(&best[4 * n + t], kb[n]);
    }
    __syncthreads();
    // block result -> grid result; the last block to finish publishes the tokens
    if (threadIdx.x < a.B) atomicMax(&a.keys[threadIdx.x], best[threadIdx.x]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
    __syncthreads();
    if (is_last) {
        __threadfence();
        const int step = *reinterpret_cast<volatile int32_t*>(a.step);
        if (threadIdx.x < a.B) {
            const int b = threadIdx.x;
            const unsigned long long k = atomicExch(&a.keys[b], 0ull);
            const int tok = (int)argmax_key_index(k);
            a.tokens[b] = tok;
            if (step < a.out_cap) a.out_ids[(size_t)b * a.out_cap + step] = tok;
            if (a.advance_pos) a.pos[b] += 1;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            *a.step = step + 1;
            *a.counter = 0u;
        }
    }
    if (!ok && threadIdx.x == 0) mbar_wait_bounded(&xbar, 0);
}

// Launch with programmatic stream serialization (see pdl_wait).
template <typename... KArgs, typename... Args>
static void launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kern, args...);
}

// The staged kernel with ks-CTA clusters (ks > 1), programmatic stream
// serialization and dyn bytes of dynamic shared memory.
template <int NT, int MODE, bool FRAG>
static bool launch_gemv_staged(const GemvArgs& a, int grid, int ks, uint32_t dyn, cudaStream_t st) {
    const void* fn = (const void*)gemv_staged_kernel<NT, MODE, FRAG>;
    if (allow_max_dynamic_smem(fn) != cudaSuccess) return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = ks;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = ks > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, gemv_staged_kernel<NT, MODE, FRAG>, a) == cudaSuccess;
}

// Shared memory above which the wide lm_head kernel is not used (bytes of
// activation planes per CTA).
constexpr uint32_t kHeadPlanesMax = 160u * 1024u;

template <int NT>
static bool launch_lm_head_wide(const GemvArgs& a, cudaStream_t st) {
    const uint32_t dyn = (uint32_t)(a.K >> 5) * NT * 512u;
    if (dyn > kHeadPlanesMax) return false;
    const void* fn = (const void*)lm_head_wide_kernel<NT>;
    if (allow_max_dynamic_smem(fn) != cudaSuccess) return false;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lm_head_wide_kernel<NT>, head_threads<NT>(), dyn) !=
            cudaSuccess ||
        per_sm < 1)
        return false;
    const int tiles = a.rows >> 4, warps = head_threads<NT>() / 32;
    const int grid = std::min(sms * per_sm, (tiles + warps - 1) / warps);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(head_threads<NT>());
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lm_head_wide_kernel<NT>, a) == cudaSuccess;
}

template <int NT>
static void launch_gemv_nt(const GemvArgs& a, int mode, int grid, cudaStream_t st) {
    if (mode == kArgmax && a.xfrag && launch_lm_head_wide<NT>(a, st)) return;
    // one CTA per (tile, K part) whose weight slice fits: the staged kernel
    const int ks = (mode == kResid && a.ksplit > 1) ? a.ksplit : 1;
    const int kpairs = a.K >> 5;
    const uint32_t dyn = (uint32_t)((kpairs + ks - 1) / ks) * 512u;
    if (mode != kArgmax && grid == (a.rows >> 4) * ks && ks <= 8 && dyn <= kGemvStageMax) {
        bool ok = false;
        if (a.xfrag) {
            switch (mode) {
                case kStore: ok = launch_gemv_staged<NT, kStore, true>(a, grid, ks, dyn, st); break;
                case kResid: ok = launch_gemv_staged<NT, kResid, true>(a, grid, ks, dyn, st); break;
                default: ok = launch_gemv_staged<NT, kSiluGate, true>(a, grid, ks, dyn, st); break;
            }
        } else {
            switch (mode) {
                case kStore: ok = launch_gemv_staged<NT, kStore, false>(a, grid, ks, dyn, st); break;
                case kResid: ok = launch_gemv_staged<NT, kResid, false>(a, grid, ks, dyn, st); break;
                default: ok = launch_gemv_staged<NT, kSiluGate, false>(a, grid, ks, dyn, st); break;
            }
        }
        if (ok) return;
    }
    switch (mode) {
        case kStore: launch_pdl(gemv_kernel<NT, kStore>, grid, 256, 0, st, a); break;
        case kResid: launch_pdl(gemv_kernel<NT, kResid>, grid, 256, 0, st, a); break;
        case kSiluGate: launch_pdl(gemv_kernel<NT, kSiluGate>, grid, 256, 0, st, a); break;
        default: launch_pdl(gemv_kernel<NT, kArgmax>, grid, 256, 0, st, a); break;
    }
}

void launch_gemv(const GemvArgs& a, int mode, int grid, cudaStream_t st) {
    const int nt = (a.B + 3) / 4;
    if (nt <= 1) launch_gemv_nt<1>(a, mode, grid, st);
    else if (nt <= 2) launch_gemv_nt<2>(a, mode, grid, st);
    else if (nt <= 4) launch_gemv_nt<4>(a, mode, grid, st);
    else launch_gemv_nt<8>(a, mode, grid, st);
}

int gemv_grid(int rows, int mode, int num_sms) {
    const int tiles = rows / 16;
    if (mode == kArgmax) return tiles < num_sms * 8 ? tiles : num_sms * 8;
    return tiles;
}

// =====================================================================
// Embedding gather from the tied int8 table: x = float(q[tok]) * s[tok].
// =====================================================================
// An id outside [0, vocab) is never dereferenced: its row is filled with
// zeros and the status word records it (the call reports invalid arguments).
__global__ void embed_kernel(const int32_t* ids, const int8_t* E, const float* sE, int H, int vocab, float* x,
                             int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    const int tok = ids[r];
    if (tok < 0 || tok >= vocab) {
        if (threadIdx.x == 0) set_status(status, kStatusBadToken);
        for (int i = threadIdx.x; i < H; i += blockDim.x) x[(size_t)r * H + i] = 0.f;
        return;
    }
    const float s = sE[tok];
    const int8_t* row = E + (size_t)tok * H;
    for (int i = threadIdx.x; i < H; i += blockDim.x) x[(size_t)r * H + i] = (float)row[i] * s;
}

void launch_embed(const int32_t* ids, int n, const int8_t* E, const float* sE, int H, int vocab, float* x,
                  int32_t* status, cudaStream_t st) {
    if (n > 0) launch_pdl(embed_kernel, n, 256, 0, st, ids, E, sE, H, vocab, x, status);
}

// =====================================================================
// RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, one row per CTA.  Writes fp32
// rows (xn, [n][H]) and/or f16 hi/lo planes (xh, columns 2i and 2i+1).
// =====================================================================
__global__ void rmsnorm_kernel(const float* x, const int32_t* rows, int H, const float* g, float eps, float* xn,
                               __half* xh, int frag) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float part[32];
    __shared__ float s_inv;
    const int i = blockIdx.x;
    const int r = rows ? rows[i] : i;
    const float* xr = x + (size_t)r * H;
    float ss = 0.f;
    for (int k = threadIdx.x; k < H; k += blockDim.x) ss += xr[k] * xr[k];
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += part[w];
        s_inv = 1.0f / sqrtf(tot / (float)H + eps);
    }
    __syncthreads();
    const float inv = s_inv;
    // a row may be spread over gridDim.y CTAs: each computes the whole sum
    // (same order) and writes its slice
    const int k_lo = (int)((long long)H * blockIdx.y / gridDim.y), k_hi = (int)((long long)H * (blockIdx.y + 1) / gridDim.y);
    for (int k = k_lo + threadIdx.x; k < k_hi; k += blockDim.x) {
        const float v = __fmul_rn(__fmul_rn(xr[k], inv), g[k]);
        if (xn) xn[(size_t)i * H + k] = v;
        if (xh) {
            __half hi, lo;
            split_f16(v, hi, lo);
            xh[plane_index(2 * i, k, H, frag)] = hi;
            xh[plane_index(2 * i + 1, k, H, frag)] = lo;
        }
    }
}

void launch_rmsnorm(const float* x, const int32_t* rows, int n, int H, const float* g, float eps, float* xn,
                    __half* xh, cudaStream_t st, int frag) {
    // few rows (decode): spread each row's writes over up to 8 CTAs, about 64 CTAs in all
    const int parts = std::max(1, std::min(std::min(8, H / 256), 64 / n));
    if (n > 0) launch_pdl(rmsnorm_kernel, dim3(n, parts), 256, 0, st, x, rows, H, g, eps, xn, xh, frag);
}

// =====================================================================
// Per-head RMSNorm on Q and K, RoPE (rotate-half, theta^(-2i/hd)), and the
// bf16 KV append at each row's position.  One warp per head; lane l holds
// elements l + 32j, so both members of every rotation pair sit in one lane.
// =====================================================================
template <int HD>
__global__ void qk_rope_append_kernel(const float* qkv, int nh, int nkv, const int32_t* row_seq,
                                      const int32_t* row_pos, const float* q_norm, const float* k_norm, float eps,
                                      const float2* rope_cs, float* q_out, __nv_bfloat16* kc, __nv_bfloat16* vc,
                                      int cap) {
    constexpr int E = HD / 32;
    const int r = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seq = row_seq[r], pos = row_pos[r];
    const int width = (nh + 2 * nkv) * HD;
    const float* row = qkv + (size_t)r * width;
    const float2* cs = rope_cs + (size_t)pos * (HD / 2);
    for (int h = warp; h < nh + nkv; h += (blockDim.x >> 5)) {
        const bool is_q = h < nh;
        const float* src = row + (size_t)h * HD;  // q heads, then k heads
        const float* gain = is_q ? q_norm : k_norm;
        float v[E];
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < E; ++j) {
            v[j] = src[lane + 32 * j];
            ss += v[j] * v[j];
        }
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
        for (int j = 0; j < E; ++j) v[j] = __fmul_rn(__fmul_rn(v[j], inv), gain[lane + 32 * j]);
#pragma unroll
        for (int j = 0; j < E / 2; ++j) {
            const float2 c = cs[lane + 32 * j];  // (cos, sin) of pair lane + 32j
            const float a0 = v[j], b0 = v[j + E / 2];
            v[j] = __fsub_rn(__fmul_rn(a0, c.x), __fmul_rn(b0, c.y));
            v[j + E / 2] = __fadd_rn(__fmul_rn(b0, c.x), __fmul_rn(a0, c.y));
        }
        if (is_q) {
            float* dst = q_out + ((size_t)r * nh + h) * HD;
#pragma unroll
            for (int j = 0; j < E; ++j) dst[lane + 32 * j] = v[j];
        } else {
            const int gk = h - nh;
            const size_t slot = (((size_t)seq * nkv + gk) * cap + pos) * HD;
            const float* vsrc = row + (size_t)(nh + nkv + gk) * HD;
#pragma unroll
            for (int j = 0; j < E; ++j) {
                kc[slot + lane + 32 * j] = __float2bfloat16_rn(v[j]);
                vc[slot + lane + 32 * j] = __float2bfloat16_rn(vsrc[lane + 32 * j]);
            }
        }
    }
}

void launch_qk_rope_append(const float* qkv, int R, int nh, int nkv, int hd, const int32_t* row_seq,
                           const int32_t* row_pos, const float* q_norm, const float* k_norm, float eps,
                           const float2* rope_cs, float* q_out, __nv_bfloat16* kc, __nv_bfloat16* vc, int cap,
                           cudaStream_t st) {
    if (R <= 0) return;
    int threads = 32 * (nh + nkv);
    if (threads > 512) threads = 512;
    if (hd == 128)
        qk_rope_append_kernel<128><<<R, threads, 0, st>>>(qkv, nh, nkv, row_seq, row_pos, q_norm, k_norm, eps,
                                                          rope_cs, q_out, kc, vc, cap);
    else
        qk_rope_append_kernel<64><<<R, threads, 0, st>>>(qkv, nh, nkv, row_seq, row_pos, q_norm, k_norm, eps,
                                                         rope_cs, q_out, kc, vc, cap);
}

// =====================================================================
// Split-KV grouped-query decode attention.
//
// CTA (split, kv head g, row r) covers a contiguous slice of the row's
// positions.  K and V are staged 64 positions at a time into shared memory
// by 1-D bulk copies (TMA) on an mbarrier, two stages deep.  The GROUP query
// heads that share kv head g are processed together, so every K/V byte is
// read once per group.  Warp w scores positions 16w..16w+15 of each chunk
// (lane l holds dims HD/32 * l ..), keeps an online softmax (running max,
// sum, weighted V), and the four warps merge their states in shared memory.
// The per-split states (acc[HD], m, l) go to `part`; the merge kernel
// combines the splits.
// =====================================================================
constexpr int kChunk = 64;

template <int HD>
struct AttnSmem {
    __nv_bfloat16 k[2][kChunk * HD];
    __nv_bfloat16 v[2][kChunk * HD];
    uint64_t bar[2];
};

// Lane layout of the chunk loop: a warp scores J positions at once with
// T = 32 / J lanes per position, each lane holding DL of the head's dims in
// pieces of P consecutive dims (16-byte pieces where DL >= 8, so that one
// load instruction of the warp reads whole 128-byte lines of a row).  With
// few query heads per group, several positions per warp step cut the
// shuffle reductions per score; the per-lane query and accumulator registers
// (GROUP * DL each) stay at 32.
template <int HD, int GROUP>
struct AttnLanes {
    static constexpr int J = GROUP <= 2 ? 4 : (GROUP <= 4 ? 2 : 1);
    static constexpr int T = 32 / J;
    static constexpr int DL = HD / T;
    static constexpr int P = DL < 8 ? DL : 8;
    // head dim of element e of lane t
    static __device__ __forceinline__ int dim(int t, int e) { return (e / P) * (T * P) + t * P + (e % P); }
};

// N consecutive bf16 (N = 2, 4 or 8; 4 N-byte aligned) -> float.
template <int N>
Q3_DEV void ld_bf16(const __nv_bfloat16* p, float* out) {
    uint32_t w[N / 2];
    if constexpr (N == 8) {
        const uint4 r = *reinterpret_cast<const uint4*>(p);
        w[0] = r.x, w[1] = r.y, w[2] = r.z, w[3] = r.w;
    } else if constexpr (N == 4) {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        w[0] = r.x, w[1] = r.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t*>(p);
    }
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        out[2 * i] = bf16_bits_to_float(w[i] & 0xffff);
        out[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
}

// The first two K/V stages of positions [start, end) (thread 0).
template <int HD>
Q3_DEV void attn_issue_first(AttnSmem<HD>& sm, const __nv_bfloat16* kb, const __nv_bfloat16* vb, int start, int end) {
    constexpr uint32_t kBytes = kChunk * HD * 2;
    const int nchunks = end > start ? (end - start + kChunk - 1) / kChunk : 0;
    for (int c = 0; c < 2 && c < nchunks; ++c) {
        mbar_arrive_expect_tx(&sm.bar[c], 2 * kBytes);
        bulk_g2s(sm.k[c], kb + (size_t)c * kChunk * HD, kBytes, &sm.bar[c]);
        bulk_g2s(sm.v[c], vb + (size_t)c * kChunk * HD, kBytes, &sm.bar[c]);
    }
}

// The chunk loop shared by the decode attention kernels: positions
// [start, end) of one (sequence, kv head) in chunks of kChunk, staged two
// at a time by bulk copies; each warp folds its 16 positions of a chunk into
// its own online-softmax state (m, l, acc) for the GROUP query heads, J
// positions per step (AttnLanes).  On return l and acc are summed over the
// warp's position lanes: every lane holds l, and the lanes of one dim group
// t hold that group's acc.  False when a bounded wait gave up (the status
// is set, copies drained).  first_issued: the caller has already issued the
// first two stages (attn_issue_first).
template <int HD, int GROUP>
Q3_DEV bool attn_chunks(AttnSmem<HD>& sm, const __nv_bfloat16* kb, const __nv_bfloat16* vb, int start, int end,
                        const float (&qr)[GROUP][AttnLanes<HD, GROUP>::DL], float scale, float (&m)[GROUP],
                        float (&l)[GROUP], float (&acc)[GROUP][AttnLanes<HD, GROUP>::DL], int32_t* status,
                        bool first_issued = false) {
    using Ln = AttnLanes<HD, GROUP>;
    constexpr int J = Ln::J, T = Ln::T, DL = Ln::DL, P = Ln::P, IT = 16 / J;
    constexpr uint32_t kBytes = kChunk * HD * 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = lane / T, t = lane % T;
    const int nchunks = end > start ? (end - start + kChunk - 1) / kChunk : 0;
    if (threadIdx.x == 0 && !first_issued) attn_issue_first<HD>(sm, kb, vb, start, end);
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (!mbar_wait_bounded(&sm.bar[s], (c >> 1) & 1)) {
            ok = false;
            break;
        }
        const int p0 = start + c * kChunk + warp * 16 + j;  // this lane's first position
        float sc[GROUP][IT];
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const __nv_bfloat16* krow = sm.k[s] + (size_t)(warp * 16 + it * J + j) * HD;
            float kv[DL];
#pragma unroll
            for (int e = 0; e < DL; e += P) ld_bf16<P>(krow + Ln::dim(t, e), kv + e);
#pragma unroll
            for (int h = 0; h < GROUP; ++h) {
                float dot = 0.f;
#pragma unroll
                for (int d = 0; d < DL; ++d) dot += qr[h][d] * kv[d];
#pragma unroll
                for (int o = 1; o < T; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                sc[h][it] = (p0 + it * J < end) ? dot * scale : -INFINITY;
            }
        }
        float pr[GROUP][IT];
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
            float cm = sc[h][0];
#pragma unroll
            for (int it = 1; it < IT; ++it) cm = fmaxf(cm, sc[h][it]);
#pragma unroll
            for (int o = T; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            const float mn = fmaxf(m[h], cm);  // -inf only while the state is still empty
            const float corr = (m[h] == -INFINITY) ? 0.f : expf(m[h] - mn);
            l[h] *= corr;
#pragma unroll
            for (int d = 0; d < DL; ++d) acc[h][d] *= corr;
#pragma unroll
            for (int it = 0; it < IT; ++it) pr[h][it] = (sc[h][it] == -INFINITY) ? 0.f : expf(sc[h][it] - mn);
            m[h] = mn;
        }
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const __nv_bfloat16* vrow = sm.v[s] + (size_t)(warp * 16 + it * J + j) * HD;
            float vv[DL];
#pragma unroll
            for (int e = 0; e < DL; e += P) ld_bf16<P>(vrow + Ln::dim(t, e), vv + e);
#pragma unroll
            for (int h = 0; h < GROUP; ++h) {
                l[h] += pr[h][it];
#pragma unroll
                for (int d = 0; d < DL; ++d) acc[h][d] += pr[h][it] * vv[d];
            }
        }
        __syncthreads();  // every warp is done with stage s
        if (threadIdx.x == 0 && c + 2 < nchunks) {
            mbar_arrive_expect_tx(&sm.bar[s], 2 * kBytes);
            bulk_g2s(sm.k[s], kb + (size_t)(c + 2) * kChunk * HD, kBytes, &sm.bar[s]);
            bulk_g2s(sm.v[s], vb + (size_t)(c + 2) * kChunk * HD, kBytes, &sm.bar[s]);
        }
    }
    // sum the position lanes (j) of l and acc
#pragma unroll
    for (int o = T; o < 32; o <<= 1)
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
            l[h] += __shfl_xor_sync(0xffffffffu, l[h], o);
#pragma unroll
            for (int d = 0; d < DL; ++d) acc[h][d] += __shfl_xor_sync(0xffffffffu, acc[h][d], o);
        }
    if (!ok && threadIdx.x == 0) {
        // a bounded wait gave up: record it and give the other copy a bounded chance to land
        set_status(status, kStatusTimeout);
        for (int s = 0; s < 2; ++s) mbar_wait_bounded(&sm.bar[s], 0);
    }
    return ok;
}

// Merge the four warps' online-softmax states and write this split's
// partial state {acc[HD], m, l} per query head; or, when outh is given (the
// only split of its row), the attention output acc / l itself as hi/lo f16
// planes, row r, query heads h0.. (the merge kernel's arithmetic for one
// split, whose weight e^0 is exactly 1).
template <int HD, int GROUP>
Q3_DEV void attn_write_partial(const float (&m)[GROUP], const float (&l)[GROUP],
                               const float (&acc)[GROUP][AttnLanes<HD, GROUP>::DL], float (&wm)[4][GROUP],
                               float (&wl)[4][GROUP], float (&wacc)[4][GROUP][HD], float* outp, int splits, int sp,
                               __half* outh = nullptr, int ldh = 0, int frag = 0, int r = 0, int h0 = 0) {
    using Ln = AttnLanes<HD, GROUP>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        for (int h = 0; h < GROUP; ++h) {
            wm[warp][h] = m[h];
            wl[warp][h] = l[h];
        }
    if (lane < Ln::T)  // position lane 0 of each dim group
#pragma unroll
        for (int h = 0; h < GROUP; ++h)
#pragma unroll
            for (int e = 0; e < Ln::DL; ++e) wacc[warp][h][Ln::dim(lane, e)] = acc[h][e];
    __syncthreads();
    for (int i = threadIdx.x; i < GROUP * HD; i += blockDim.x) {
        const int h = i / HD, d = i % HD;
        float M = -INFINITY;
        for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w][h]);
        float L = 0.f, A = 0.f;
        for (int w = 0; w < 4; ++w) {
            if (wm[w][h] == -INFINITY) continue;
            const float f = expf(wm[w][h] - M);
            L += wl[w][h] * f;
            A += wacc[w][h][d] * f;
        }
        if (outh) {
            __half hi, lo;
            split_f16(A / L, hi, lo);
            outh[plane_index(2 * r, (h0 + h) * HD + d, ldh, frag)] = hi;
            outh[plane_index(2 * r + 1, (h0 + h) * HD + d, ldh, frag)] = lo;
            continue;
        }
        float* o = outp + ((size_t)h * splits + sp) * (HD + 2);
        o[d] = A;
        if (d == 0) {
            o[HD] = M;
            o[HD + 1] = L;
        }
    }
}

// Split s of row r attends positions [start, end) of its sequence with
// queries that are already normed and rotated.
template <int HD, int GROUP>
__global__ void __launch_bounds__(128) attn_split_kernel(const float* q, const __nv_bfloat16* kc,
                                                         const __nv_bfloat16* vc, const int32_t* row_seq,
                                                         const int32_t* row_len, int len_add, int nh, int nkv,
                                                         int cap, int splits, float* part, int32_t* status) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    AttnSmem<HD>& sm = *reinterpret_cast<AttnSmem<HD>*>(smem_raw);
    __shared__ float wm[4][GROUP], wl[4][GROUP];
    __shared__ float wacc[4][GROUP][HD];

    const int sp = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int lane = threadIdx.x & 31;
    const int len = row_len[r] + len_add, seq = row_seq[r];
    int per = (len + splits - 1) / splits;
    per = (per + kChunk - 1) / kChunk * kChunk;
    const int start = sp * per;
    const int end = min(len, start + per);
    float* outp = part + ((size_t)r * nh + (size_t)g * GROUP) * splits * (HD + 2);
    if (start >= end) {
        for (int i = threadIdx.x; i < GROUP * (HD + 2); i += blockDim.x) {
            const int h = i / (HD + 2), e = i % (HD + 2);
            outp[((size_t)h * splits + sp) * (HD + 2) + e] = (e == HD) ? -INFINITY : 0.f;
        }
        return;
    }
    const size_t head_base = ((size_t)seq * nkv + g) * cap * HD;
    if (threadIdx.x == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();

    using Ln = AttnLanes<HD, GROUP>;
    constexpr int D = Ln::DL;
    const int t = lane % Ln::T;
    float qr[GROUP][D];
#pragma unroll
    for (int h = 0; h < GROUP; ++h)
#pragma unroll
        for (int d = 0; d < D; ++d) qr[h][d] = q[((size_t)r * nh + g * GROUP + h) * HD + Ln::dim(t, d)];
    const float scale = 1.0f / sqrtf((float)HD);
    float m[GROUP], l[GROUP], acc[GROUP][D];
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) acc[h][d] = 0.f;
    }
    if (!attn_chunks<HD, GROUP>(sm, kc + head_base + (size_t)start * HD, vc + head_base + (size_t)start * HD, start,
                                end, qr, scale, m, l, acc, status))
        return;
    attn_write_partial<HD, GROUP>(m, l, acc, wm, wl, wacc, outp, splits, sp);
}

// The decode attention's balanced split plan.  Row r of the step (len_r =
// row_pos[r] + 1 positions, R <= 32 rows) gets s_r = ceil(len_r / P) splits
// of P positions, P the smallest multiple of kChunk with sum_r s_r <= G and
// every s_r <= smax (G >= R): long rows take more CTAs than short ones and
// every split is at most P long.  Evaluated by one whole warp; every lane
// returns P.
Q3_DEV int plan_split_len(const int32_t* row_pos, int R, int G, int smax, int cap) {
    const int lane = threadIdx.x & 31;
    const int len = lane < R ? row_pos[lane] + 1 : 0;
    const int total = __reduce_add_sync(0xffffffffu, len);
    const int maxlen = __reduce_max_sync(0xffffffffu, len);
    int P = max((total + G - 1) / G, (maxlen + smax - 1) / smax);
    P = max(kChunk, (P + kChunk - 1) / kChunk * kChunk);
#pragma unroll 1
    for (int it = 0; it <= cap / kChunk; ++it) {  // P >= maxlen fits (G >= R)
        if (__reduce_add_sync(0xffffffffu, (len + P - 1) / P) <= G) break;
        P += kChunk;
    }
    return P;
}

// CTA `i` of a kv head under the plan: its row (or -1 when the rows need
// fewer than i + 1 splits), its split index and its row's split count.
Q3_DEV void plan_cta(const int32_t* row_pos, int R, int P, int i, int& r, int& sp, int& nr) {
    const int lane = threadIdx.x & 31;
    const int s = lane < R ? (row_pos[lane] + 1 + P - 1) / P : 0;
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int excl = incl - s;
    const unsigned hit = __ballot_sync(0xffffffffu, s > 0 && excl <= i && i < incl);
    r = hit ? __ffs(hit) - 1 : -1;
    sp = r >= 0 ? i - __shfl_sync(0xffffffffu, excl, r) : 0;
    nr = r >= 0 ? __shfl_sync(0xffffffffu, s, r) : 0;
}

// Whether the decode attention asks L2 for its cached K/V before waiting on
// the previous kernel.
constexpr bool kAttnPrefetch = true;

// Decode step with the QK-RMSNorm, RoPE and KV append folded in: row r's new
// position p = row_pos[r] is appended (bf16, by the split that owns p) and
// attended from registers, so the cache reads cover positions < p only.
template <int HD, int GROUP>
__global__ void __launch_bounds__(128) attn_decode_kernel(const float* qkv, const float* q_norm, const float* k_norm,
                                                          float eps, const float2* rope_cs, __nv_bfloat16* kc,
                                                          __nv_bfloat16* vc, const int32_t* row_seq,
                                                          const int32_t* row_pos, int nh, int nkv, int cap,
                                                          int G, int R, int smax, float* part, __half* outh,
                                                          int ldh, int frag, int32_t* status) {
    pdl_launch_dependents();
    using Ln = AttnLanes<HD, GROUP>;
    constexpr int D = Ln::DL;
    constexpr int E = HD / 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    AttnSmem<HD>& sm = *reinterpret_cast<AttnSmem<HD>*>(smem_raw);
    __shared__ float wm[4][GROUP], wl[4][GROUP];
    __shared__ float wacc[4][GROUP][HD];
    __shared__ float qs[GROUP][HD], kp[HD], vp[HD];
    __shared__ int s_plan[4];  // P, row, split, the row's splits

    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The positions and the cached K/V of positions < pos are final here:
    // the previous launch lets this one start only after its own wait, when
    // every launch before it has completed.  The split plan is made now and
    // the first two stages are issued before the wait.
    if (warp == 0) {
        const int P = plan_split_len(row_pos, R, G, smax, cap);
        int pr, psp, pnr;
        plan_cta(row_pos, R, P, blockIdx.x, pr, psp, pnr);
        if (lane == 0) s_plan[0] = P, s_plan[1] = pr, s_plan[2] = psp, s_plan[3] = pnr;
    }
    __syncthreads();
    const int P = s_plan[0], r = s_plan[1], sp = s_plan[2], nr = s_plan[3];
    if (r < 0) return;  // the rows need fewer splits than this kv head has CTAs
    const int pos = row_pos[r], seq = row_seq[r];
    const int len = pos + 1;
    const int start = sp * P;
    const int end = min(len, start + P);  // non-empty: sp < ceil(len / P)
    const bool owns_p = pos >= start && pos < end;
    const int cend = owns_p ? pos : end;  // cached positions only
    const size_t head_base = ((size_t)seq * nkv + g) * cap * HD;
    if (threadIdx.x == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
        attn_issue_first<HD>(sm, kc + head_base + (size_t)start * HD, vc + head_base + (size_t)start * HD, start,
                             cend);
    }
    if (kAttnPrefetch) {
        // the rest of the split: asked of L2
        const int lo = start + 2 * kChunk;
        if (lo < cend) {
            const size_t base = head_base + (size_t)lo * HD;
            const uint32_t bytes = (uint32_t)(cend - lo) * HD * 2u;
            for (uint32_t off = threadIdx.x * 4096u; off < bytes; off += blockDim.x * 4096u) {
                const uint32_t n = bytes - off < 4096u ? bytes - off : 4096u;
                prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(kc + base) + off, n);
                prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(vc + base) + off, n);
            }
        }
    }
    pdl_wait();
    float* outp = part + ((size_t)r * nh + (size_t)g * GROUP) * smax * (HD + 2);

    // the group's queries (and, in the owning split, the new K and V): one
    // warp per head, lane l holding elements l + 32j
    const float* row = qkv + (size_t)r * (nh + 2 * nkv) * HD;
    const float2* cs = rope_cs + (size_t)pos * (HD / 2);
    for (int h = warp; h < GROUP + (owns_p ? 2 : 0); h += 4) {
        const bool is_v = h == GROUP + 1;
        const float* src = h < GROUP ? row + (size_t)(g * GROUP + h) * HD
                                     : row + (size_t)((is_v ? nh + nkv : nh) + g) * HD;
        float v[E];
#pragma unroll
        for (int j = 0; j < E; ++j) v[j] = src[lane + 32 * j];
        if (!is_v) {
            const float* gain = h < GROUP ? q_norm : k_norm;
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < E; ++j) ss += v[j] * v[j];
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
            for (int j = 0; j < E; ++j) v[j] = __fmul_rn(__fmul_rn(v[j], inv), gain[lane + 32 * j]);
#pragma unroll
            for (int j = 0; j < E / 2; ++j) {
                const float2 c = cs[lane + 32 * j];
                const float a0 = v[j], b0 = v[j + E / 2];
                v[j] = __fsub_rn(__fmul_rn(a0, c.x), __fmul_rn(b0, c.y));
                v[j + E / 2] = __fadd_rn(__fmul_rn(b0, c.x), __fmul_rn(a0, c.y));
            }
        }
        if (h < GROUP) {
#pragma unroll
            for (int j = 0; j < E; ++j) qs[h][lane + 32 * j] = v[j];
        } else {
            __nv_bfloat16* dst = (is_v ? vc : kc) + head_base + (size_t)pos * HD;
            float* keep = is_v ? vp : kp;
#pragma unroll
            for (int j = 0; j < E; ++j) {
                const __nv_bfloat16 b = __float2bfloat16_rn(v[j]);
                dst[lane + 32 * j] = b;
                keep[lane + 32 * j] = __bfloat162float(b);
            }
        }
    }
    __syncthreads();

    const int t = lane % Ln::T;
    float qr[GROUP][D];
#pragma unroll
    for (int h = 0; h < GROUP; ++h)
#pragma unroll
        for (int d = 0; d < D; ++d) qr[h][d] = qs[h][Ln::dim(t, d)];
    const float scale = 1.0f / sqrtf((float)HD);
    float m[GROUP], l[GROUP], acc[GROUP][D];
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) acc[h][d] = 0.f;
    }
    if (!attn_chunks<HD, GROUP>(sm, kc + head_base + (size_t)start * HD, vc + head_base + (size_t)start * HD, start,
                                cend, qr, scale, m, l, acc, status, true))
        return;
    if (owns_p && warp == 0) {
        // position p from the rounded values kept in shared memory (every
        // position lane of a dim group holds the same state)
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < D; ++d) dot += qr[h][d] * kp[Ln::dim(t, d)];
#pragma unroll
            for (int o = 1; o < Ln::T; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            const float sc = dot * scale;
            const float mn = fmaxf(m[h], sc);
            const float corr = (m[h] == -INFINITY) ? 0.f : expf(m[h] - mn);
            const float pe = expf(sc - mn);
            l[h] = l[h] * corr + pe;
#pragma unroll
            for (int d = 0; d < D; ++d) acc[h][d] = acc[h][d] * corr + pe * vp[Ln::dim(t, d)];
            m[h] = mn;
        }
    }
    attn_write_partial<HD, GROUP>(m, l, acc, wm, wl, wacc, outp, smax, sp, nr == 1 ? outh : nullptr, ldh, frag, r,
                                  g * GROUP);
}

// out[r][h][:] = sum_s acc_s e^{m_s - M} / sum_s l_s e^{m_s - M} over the
// row's non-empty splits (the split kernels' range rule); the split weights
// are computed once per block by warp 0, then every thread sums its column
// (loads batched eight splits at a time; the sum stays in split order).
template <int HD>
__global__ void attn_merge_kernel(const float* part, int nh, int splits, const int32_t* row_len, int len_add,
                                  float* out, __half* outh, int ldh, int frag, int plan_G, int plan_R,
                                  int plan_cap) {
    pdl_launch_dependents();
    __shared__ float sm_m[64], sm_f[64];
    __shared__ float s_l;
    __shared__ int s_per;
    const int rh = blockIdx.x;  // r * nh + h
    const int d = threadIdx.x;
    const int r = rh / nh, h = rh % nh;
    int nne;
    if (plan_G > 0) {
        // the decode attention's balanced plan (row_len = positions, len_add =
        // 1), made before the wait as the attention makes it: the positions
        // are final once the attention has started.  A row of one split has
        // had its output written by the attention (every CTA still waits, so
        // this launch cannot complete before the attention)
        if (d < 32) {
            const int P = plan_split_len(row_len, plan_R, plan_G, splits, plan_cap);
            if (d == 0) s_per = P;
        }
        __syncthreads();
        nne = (row_len[r] + len_add + s_per - 1) / s_per;
        pdl_wait();
        if (nne == 1) return;
    } else {
        pdl_wait();
        const int len = row_len[r] + len_add;
        int per = (len + splits - 1) / splits;
        per = (per + kChunk - 1) / kChunk * kChunk;
        nne = min(splits, (len + per - 1) / per);
    }
    const float* p = part + (size_t)rh * splits * (HD + 2);
    if (d < 32) {
        // lane j holds splits j and j + 32
        const float m0 = d < nne ? p[(size_t)d * (HD + 2) + HD] : -INFINITY;
        const float m1 = d + 32 < nne ? p[(size_t)(d + 32) * (HD + 2) + HD] : -INFINITY;
        const float M = warp_max(fmaxf(m0, m1));
        const float f0 = m0 == -INFINITY ? 0.f : expf(m0 - M);
        const float f1 = m1 == -INFINITY ? 0.f : expf(m1 - M);
        const float l0 = f0 != 0.f ? p[(size_t)d * (HD + 2) + HD + 1] * f0 : 0.f;
        const float l1 = f1 != 0.f ? p[(size_t)(d + 32) * (HD + 2) + HD + 1] * f1 : 0.f;
        const float L = warp_sum(l0 + l1);
        if (d < nne) sm_m[d] = m0, sm_f[d] = f0;
        if (d + 32 < nne) sm_m[d + 32] = m1, sm_f[d + 32] = f1;
        if (d == 0) s_l = L;
    }
    __syncthreads();
    float A = 0.f;
    for (int s0 = 0; s0 < nne; s0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = s0 + u < nne ? p[(size_t)(s0 + u) * (HD + 2) + d] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (s0 + u < nne && sm_m[s0 + u] != -INFINITY) A += v[u] * sm_f[s0 + u];
    }
    const float o = A / s_l;
    if (out) out[(size_t)rh * HD + d] = o;
    if (outh) {
        __half hi, lo;
        split_f16(o, hi, lo);
        outh[plane_index(2 * r, h * HD + d, ldh, frag)] = hi;
        outh[plane_index(2 * r + 1, h * HD + d, ldh, frag)] = lo;
    }
}

size_t attn_part_bytes(int R, int nh, int hd, int splits) { return (size_t)R * nh * splits * (hd + 2) * sizeof(float); }

template <int HD, int GROUP>
static bool launch_attn_t(const float* q, const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* row_seq,
                          const int32_t* row_len, int len_add, int R, int nh, int nkv, int cap, int splits,
                          float* part, int32_t* status, cudaStream_t st) {
    const int smem = (int)sizeof(AttnSmem<HD>);
    if (allow_max_dynamic_smem((const void*)attn_split_kernel<HD, GROUP>) != cudaSuccess) return false;
    dim3 grid(splits, nkv, R);
    attn_split_kernel<HD, GROUP><<<grid, 128, smem, st>>>(q, k, v, row_seq, row_len, len_add, nh, nkv, cap, splits,
                                                          part, status);
    return true;
}

int launch_attention(const float* q, const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* row_seq,
                     const int32_t* row_len, int len_add, int R, int nh, int nkv, int hd, int cap, int splits,
                     float* part, float* out, __half* outh, int ldh, int32_t* status, cudaStream_t st,
                     int frag) {
    if (R <= 0) return 0;
    const int group = nh / nkv;
#define Q3_ATTN_CASE(HDV, GV)                                                                         \
    if (hd == HDV && group == GV) {                                                                   \
        if (!launch_attn_t<HDV, GV>(q, k, v, row_seq, row_len, len_add, R, nh, nkv, cap, splits, part, status, \
                                    st))                                                              \
            return -2;                                                                                \
        attn_merge_kernel<HDV><<<R * nh, HDV, 0, st>>>(part, nh, splits, row_len, len_add, out, outh, ldh, \
                                                       frag, 0, 0, 0);                                        \
        return 0;                                                                                     \
    }
    Q3_ATTN_CASE(128, 1)
    Q3_ATTN_CASE(128, 2)
    Q3_ATTN_CASE(128, 4)
    Q3_ATTN_CASE(128, 8)
    Q3_ATTN_CASE(64, 1)
    Q3_ATTN_CASE(64, 2)
    Q3_ATTN_CASE(64, 4)
    Q3_ATTN_CASE(64, 8)
#undef Q3_ATTN_CASE
    return -1;  // unsupported head_dim / group
}

template <int HD, int GROUP>
static bool launch_attn_decode_t(const float* qkv, const float* q_norm, const float* k_norm, float eps,
                                 const float2* rope_cs, __nv_bfloat16* kc, __nv_bfloat16* vc, const int32_t* row_seq,
                                 const int32_t* row_pos, int R, int nh, int nkv, int cap, int G, int smax,
                                 float* part, __half* outh, int ldh, int frag, int32_t* status, cudaStream_t st) {
    const int smem = (int)sizeof(AttnSmem<HD>);
    if (allow_max_dynamic_smem((const void*)attn_decode_kernel<HD, GROUP>) != cudaSuccess) return false;
    dim3 grid(G, nkv, 1);
    launch_pdl(attn_decode_kernel<HD, GROUP>, grid, 128, smem, st, qkv, q_norm, k_norm, eps, rope_cs, kc, vc, row_seq,
               row_pos, nh, nkv, cap, G, R, smax, part, outh, ldh, frag, status);
    return true;
}

template <int HD, int GROUP>
static int attn_decode_occupancy() {
    if (allow_max_dynamic_smem((const void*)attn_decode_kernel<HD, GROUP>) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<HD, GROUP>, 128,
                                                      sizeof(AttnSmem<HD>)) != cudaSuccess)
        return 0;
    return n;
}

int attention_decode_blocks_per_sm(int hd, int group) {
#define Q3_ATTN_CASE(HDV, GV) \
    if (hd == HDV && group == GV) return attn_decode_occupancy<HDV, GV>();
    Q3_ATTN_CASE(128, 1)
    Q3_ATTN_CASE(128, 2)
    Q3_ATTN_CASE(128, 4)
    Q3_ATTN_CASE(128, 8)
    Q3_ATTN_CASE(64, 1)
    Q3_ATTN_CASE(64, 2)
    Q3_ATTN_CASE(64, 4)
    Q3_ATTN_CASE(64, 8)
#undef Q3_ATTN_CASE
    return 0;
}

int launch_attention_decode(const float* qkv, const float* q_norm, const float* k_norm, float eps,
                            const float2* rope_cs, __nv_bfloat16* kc, __nv_bfloat16* vc, const int32_t* row_seq,
                            const int32_t* row_pos, int R, int nh, int nkv, int hd, int cap, int G, int smax,
                            float* part, __half* outh, int ldh, int32_t* status, cudaStream_t st, int frag) {
    if (R <= 0) return 0;
    if (R > 32 || G < R || smax < 1 || smax > 64) return -3;
    const int group = nh / nkv;
#define Q3_ATTN_CASE(HDV, GV)                                                                                      \
    if (hd == HDV && group == GV) {                                                                                \
        if (!launch_attn_decode_t<HDV, GV>(qkv, q_norm, k_norm, eps, rope_cs, kc, vc, row_seq, row_pos, R, nh, nkv,  \
                                           cap, G, smax, part, outh, ldh, frag, status, st))                      \
            return -2;                                                                                             \
        if (G > R) /* some row may have more than one split */                                                    \
            launch_pdl(attn_merge_kernel<HDV>, R * nh, HDV, 0, st, part, nh, smax, row_pos, 1, (float*)nullptr,   \
                       outh, ldh, frag, G, R, cap);                                                                \
        return 0;                                                                                                  \
    }
    Q3_ATTN_CASE(128, 1)
    Q3_ATTN_CASE(128, 2)
    Q3_ATTN_CASE(128, 4)
    Q3_ATTN_CASE(128, 8)
    Q3_ATTN_CASE(64, 1)
    Q3_ATTN_CASE(64, 2)
    Q3_ATTN_CASE(64, 4)
    Q3_ATTN_CASE(64, 8)
#undef Q3_ATTN_CASE
    return -1;
}


}  // namespace q3
