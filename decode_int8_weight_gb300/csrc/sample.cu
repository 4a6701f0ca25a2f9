// Seeded sampling chain on the device (sm_103a).
//
// "Model-agnostic LLM inference", section "Sampling": with temperature > 0
// each token is drawn through repetition / presence / frequency penalties ->
// temperature -> top-k -> min-p -> top-p -> a seeded weighted draw; the same
// seed gives the same tokens and top_k = 1 gives the greedy sequence.  The
// page names the steps only; the readings taken here:
//   * penalties over the tokens already in the sequence (prompt and earlier
//     generated tokens), token t seen c times: a positive logit is divided by
//     the repetition penalty r and any other multiplied by it; then the
//     presence penalty and c times the frequency penalty are subtracted;
//   * the temperature divides the penalised logits;
//   * candidates are ordered by value (descending), ties by token id
//     (ascending); top-k keeps the first k;
//   * min-p keeps candidates whose softmax probability (over the candidates
//     it is given) is at least min_p times the largest;
//   * top-p keeps the shortest prefix whose softmax probabilities sum to at
//     least top_p;
//   * the draw u in [0, 1) is the top 24 bits of SplitMix64 output c + 1 from
//     the seed, c = step * 2^20 + sequence (Steele, Lea and Flood, "Fast
//     splittable pseudorandom number generators", OOPSLA 2014), and the token
//     is the first survivor whose cumulative probability exceeds u.
// Everything after the model's fp32 logits is float64 without contracted
// multiply-adds, in fixed orders, so a seed reproduces its tokens bit for bit.
//
// Layout of the work: one cluster of 8 CTAs per sequence, CTA r owning a
// contiguous eighth of the vocabulary and each of its 32 warps a contiguous
// span of that.  The k-th largest value is found by radix selection over
// 64-bit order keys of the float64 values, 12 bits a round: every CTA counts
// digits into its own shared-memory histogram and reads its peers' over
// distributed shared memory, so all 8 take the same decision.  After the
// first round only the keys sharing its digit (the "band") are kept, in
// per-warp lists in token order; later rounds read those lists, and once at
// most 64 keys in the cluster share the digits found so far, CTA 0 sorts
// those and takes what is still needed.  Each CTA sorts its candidates and
// computes their exponentials; CTA 0 gathers the 8 sorted runs, merges them
// (binary search of each candidate's place) and finishes the chain: prefix
// sums, min-p, top-p, the draw.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sample.h"

namespace cg = cooperative_groups;

namespace q3 {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;                            // 12-bit digits
constexpr int kGroups = 64, kGroupBins = kBins / kGroups;  // digits merged across the cluster group by group
constexpr int kSmallN = 256;                           // candidates one warp finishes alone
constexpr int kPerThread = kSampleMaxTopK / kThreads;  // sorted elements a thread owns in the scans

// Tokens per CTA: a multiple of 1024 so that each warp's span is a multiple of 32.
__host__ __device__ inline int band_chunk(int V) {
    return (V + kSampleCtas * 1024 - 1) / (kSampleCtas * 1024) * 1024;
}

Q3_DEV uint64_t splitmix64_output(uint64_t seed, uint64_t n) {
    uint64_t x = seed + n * 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

Q3_DEV double uniform_draw(uint64_t seed, uint32_t sequence, uint32_t step) {
    const uint64_t c = (uint64_t)step * (1ull << 20) + sequence;
    return (double)(splitmix64_output(seed, c + 1) >> 40) * 0x1p-24;
}

// Order key of float64 bits: a larger value gets a larger key; -0 and +0
// share one key.
Q3_DEV uint64_t order_key_bits(uint64_t u) {
    if ((u << 1) == 0) return 0x8000000000000000ull;
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// The order key of (double)f for an fp32 f, from its bits: the float64
// pipe of this part is narrow, and most of the vocabulary needs no other
// arithmetic.
__device__ __noinline__ uint64_t order_key_f32_rare(uint32_t b);

Q3_DEV uint64_t order_key_f32(uint32_t b) {
    const uint32_t e = (b >> 23) & 0xFFu;
    if (e == 0u || e == 0xFFu) return order_key_f32_rare(b);
    // normal: exponent rebias 1023 - 127, mantissa moved up 29 bits
    const uint64_t mag = ((uint64_t)(b & 0x7FFFFFFFu) << 29) + (896ull << 52);
    return (b >> 31) ? (~mag & 0x7FFFFFFFFFFFFFFFull) : (mag | 0x8000000000000000ull);
}

// Zero, subnormal, infinite and nan inputs of order_key_f32.
__device__ __noinline__ uint64_t order_key_f32_rare(uint32_t b) {
    const uint64_t sign = (uint64_t)(b >> 31) << 63;
    const uint32_t e = (b >> 23) & 0xFFu, m = b & 0x7FFFFFu;
    uint64_t mag;
    if (e == 0xFFu) {
        mag = (0x7FFull << 52) | ((uint64_t)m << 29);                 // inf, nan
    } else {
        if (m == 0) return 0x8000000000000000ull;                    // +-0
        const int top = 31 - __clz(m);                                 // subnormal: m * 2^-149
        mag = ((uint64_t)(top + 874) << 52) | (((uint64_t)m << (52 - top)) & 0xFFFFFFFFFFFFFull);
    }
    return order_key_bits(sign | mag);
}

// A logit after the penalties, token seen c > 0 times (float64, no
// contracted multiply-adds).  Out of line: few tokens take it.
__device__ __noinline__ double penalised(float zf, int c, const SampleParams& p) {
    double v = (double)zf;
    if (p.repeat_penalty != 1.0) v = v > 0.0 ? __ddiv_rn(v, p.repeat_penalty) : __dmul_rn(v, p.repeat_penalty);
    return __dsub_rn(__dsub_rn(v, p.presence_penalty), __dmul_rn(p.frequency_penalty, (double)c));
}

// The candidate order key of a token: its penalised logit's (the order of
// the temperature-scaled logits, since the temperature is positive).
// key_value inverts it.
Q3_DEV uint64_t token_key(float zf, int c, const SampleParams& p) {
    return c > 0 ? order_key_bits((uint64_t)__double_as_longlong(penalised(zf, c, p)))
                 : order_key_f32(__float_as_uint(zf));
}

Q3_DEV double key_value(uint64_t key) {
    return __longlong_as_double((long long)((key >> 63) ? (key & 0x7FFFFFFFFFFFFFFFull) : ~key));
}

Q3_DEV unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Inclusive prefix sums out[i] = in[0] + .. + in[i], i < n <= kSampleMaxTopK:
// thread t sums its kPerThread consecutive elements, then the threads' sums
// are scanned in order.
__device__ __noinline__ void block_inclusive_scan(const double* in, double* out, int n, double* s_w) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double own[kPerThread];
    double run = 0.0;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const int i = tid * kPerThread + j;
        run += i < n ? in[i] : 0.0;
        own[j] = run;
    }
    double incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        double x = s_w[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        s_w[lane] = x;
    }
    __syncthreads();
    const double base = (warp ? s_w[warp - 1] : 0.0) + (incl - run);
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const int i = tid * kPerThread + j;
        if (i < n) out[i] = base + own[j];
    }
    __syncthreads();
}

// First i < n with pred(w[i]) (n when none).
template <typename Pred>
Q3_DEV int block_first(const double* w, int n, Pred pred, int* s_first) {
    if (threadIdx.x == 0) *s_first = n;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads)
        if (pred(w[i])) atomicMin(s_first, i);
    __syncthreads();
    const int r = *s_first;
    __syncthreads();
    return r;
}

constexpr int kSubMax = 64;  // keys sharing the last prefix that CTA 0 sorts itself (early finish)

struct __align__(16) SampleSmem {
    uint64_t key[kSampleMaxTopK];  // this CTA's candidates, sorted before the gather (CTA 0: every CTA's runs)
    double e[kSampleMaxTopK];      // exp(v - v_max) of each candidate, v its temperature-scaled logit
    double w[kSampleMaxTopK];      // CTA 0: e in the merged order
    int hist[2][kBins];            // digit counts of even / odd rounds (CTA 0's tail: the merged tokens)
    int gsum[2][kGroups];          // their sums per group of kGroupBins digits
    int tok[kSampleMaxTopK];
    uint64_t sub_key[kSubMax];     // early finish: keys sharing the prefix (CTA 0: the cluster's)
    int sub_tok[kSubMax];
    int tie_before[kWarps];
    int run_off[kSampleCtas + 1];  // CTA 0: where each CTA's run starts after the gather
    double dbl[kWarps];
    unsigned long long kmax;       // this CTA's largest candidate key
    int n_sel;                     // entries in key / tok / e
    int n_sub;                     // entries in sub_key / sub_tok
    int ties;                      // keys equal to the k-th key in this CTA
    int digit, need, count, first;
};

// Append one candidate to this CTA's selection.
Q3_DEV void select_one(SampleSmem& s, uint64_t key, int token) {
    const int i = atomicAdd(&s.n_sel, 1);
    if (i < kSampleMaxTopK) s.key[i] = key, s.tok[i] = token;
}

// Candidate order: key descending, then token ascending.
Q3_DEV bool before(uint64_t ka, int ta, uint64_t kb, int tb) { return ka > kb || (ka == kb && ta < tb); }

// Bitonic sort of key[0..n) / tok[0..n) in candidate order over the next
// power of two (the padding sorts last), by the `nt` threads with index
// below nt; sync() is their barrier.
template <typename Sync>
Q3_DEV void bitonic(uint64_t* key, int* tok, int n, int nt, Sync sync) {
    const int tid = threadIdx.x;
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int i = n + tid; i < n2; i += nt) key[i] = 0ull, tok[i] = 0x7fffffff;
    sync();
#pragma unroll 1
    for (int size = 2; size <= n2; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += nt) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint64_t ki = key[i], kj = key[j];
                    const int ti = tok[i], tj = tok[j];
                    if (before(ki, ti, kj, tj) != ((i & size) == 0)) key[i] = kj, key[j] = ki, tok[i] = tj, tok[j] = ti;
                }
            }
            sync();
        }
    }
}

// Sort of this CTA's n candidates by all threads (warp 0 alone for n <= 64);
// ends with a block barrier.
__device__ __noinline__ void sort_candidates(uint64_t* key, int* tok, int n) {
    if (n <= 64) {
        if (threadIdx.x < 32) bitonic(key, tok, n, 32, [] { __syncwarp(); });
    } else {
        bitonic(key, tok, n, kThreads, [] { __syncthreads(); });
    }
    __syncthreads();
}

// Warp-level search of a descending run of 64 counts held two per lane
// (lane l: positions 63 - 2l and 62 - 2l): the position where the running
// count from the top reaches `need`, `need` less the counts above it, and
// the count at that position.  Returns false when the counts do not reach
// `need`.
Q3_DEV bool warp_cross64(int hi, int lo, int need, int& pos, int& rest, int& at_count) {
    const int lane = threadIdx.x & 31;
    int incl = hi + lo;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int above = incl - hi - lo;
    int at = -1, left = 0, c = 0;
    if (above < need && above + hi >= need) at = 63 - 2 * lane, left = need - above, c = hi;
    else if (above + hi < need && above + hi + lo >= need) at = 62 - 2 * lane, left = need - above - hi, c = lo;
    const unsigned who = __ballot_sync(0xffffffffu, at >= 0);
    if (!who) return false;
    const int src = __ffs(who) - 1;
    pos = __shfl_sync(0xffffffffu, at, src);
    rest = __shfl_sync(0xffffffffu, left, src);
    at_count = __shfl_sync(0xffffffffu, c, src);
    return true;
}

// One radix round's decision, taken identically by every CTA of the
// cluster: the digit d of the k-th largest key among the keys counted in
// hist[r & 1] of all 8 CTAs (the keys that match the digits found so far),
// `need` reduced by the count of keys with a larger digit, and in *count
// the number of keys with digit d.  The counts are merged in two steps to
// keep the distributed shared-memory reads small: the 64 group sums of
// every CTA, then the 64 digits of the group that holds the k-th key.  Also
// clears the other histogram for the next round (every peer finished
// reading it before arriving at this round's cluster barrier).
__device__ __noinline__ int select_digit(SampleSmem& s, int r, int& need, int* count, cg::cluster_group& cl) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __syncthreads();  // this CTA's histogram is complete
    {
        const int g = tid >> 4;
        const int4 v = reinterpret_cast<const int4*>(s.hist[r & 1] + g * kGroupBins)[tid & 15];
        int x = v.x + v.y + v.z + v.w;
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        if ((tid & 15) == 0) s.gsum[r & 1][g] = x;
    }
    cl.sync();
    for (int i = tid; i < kBins; i += kThreads) s.hist[(r + 1) & 1][i] = 0;
    if (warp == 0) {
        int hi = 0, lo = 0;
#pragma unroll
        for (int peer = 0; peer < kSampleCtas; ++peer) {
            const int* pg = cl.map_shared_rank(s.gsum[r & 1], peer);
            hi += pg[63 - 2 * lane], lo += pg[62 - 2 * lane];
        }
        int g = 0, rest = need, gc = 0;
        if (warp_cross64(hi, lo, need, g, rest, gc)) {
            hi = lo = 0;
#pragma unroll
            for (int peer = 0; peer < kSampleCtas; ++peer) {
                const int* ph = cl.map_shared_rank(s.hist[r & 1], peer) + g * kGroupBins;
                hi += ph[63 - 2 * lane], lo += ph[62 - 2 * lane];
            }
            int d = 0, left = rest, dc = 0;
            if (warp_cross64(hi, lo, rest, d, left, dc) && lane == 0)
                s.digit = g * kGroupBins + d, s.need = left, s.count = dc;
        }
    }
    __syncthreads();
    need = s.need;
    *count = s.count;
    return s.digit;
}

// Prefix sums cum[i] = ew[0] + .. + ew[i] of the n candidates in order, then
// min-p, top-p and the draw u01 in [0, 1): the index of the drawn candidate.
// Compared on unnormalised sums: the softmax over the first m candidates is
// ew[i] / cum[m - 1].  Warp 0 alone (lane l owning elements 8l .. 8l + 7)
// for n <= kSmallN; the whole block otherwise.
__device__ __noinline__ int finish_small(const double* ew, double* cum, int n, const SampleParams& p, double u01) {
    const int lane = threadIdx.x & 31;
    constexpr int kOwn = kSmallN / 32;
    double own[kOwn];
    double run = 0.0;
#pragma unroll
    for (int j = 0; j < kOwn; ++j) {
        const int i = kOwn * lane + j;
        run += i < n ? ew[i] : 0.0;
        own[j] = run;
    }
    double incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
#pragma unroll
    for (int j = 0; j < kOwn; ++j) {
        const int i = kOwn * lane + j;
        if (i < n) cum[i] = (incl - run) + own[j];
    }
    __syncwarp();
    auto first = [&](const double* a, int m, auto pred) {  // first i < m with pred(a[i]), else m
        int f = m;
        for (int j = 0; j < kOwn; ++j) {
            const int i = kOwn * lane + j;
            if (i < m && pred(a[i])) {
                f = i;
                break;
            }
        }
        return (int)__reduce_min_sync(0xffffffffu, (unsigned)f);
    };
    int m = n;
    if (p.min_p > 0.0) {  // probability at least min_p times the largest (candidate 0's)
        const double floor_e = p.min_p * ew[0];
        m = max(1, first(ew, m, [&](double e) { return !(e >= floor_e); }));
    }
    if (p.top_p < 1.0) {  // the shortest prefix whose probabilities sum to at least top_p
        const double want = p.top_p * cum[m - 1];
        m = min(m, 1 + first(cum, m, [&](double c) { return c >= want; }));
    }
    const double u = u01 * cum[m - 1];  // the first survivor whose cumulative probability exceeds u
    return min(m - 1, first(cum, m, [&](double c) { return u < c; }));
}

__device__ __noinline__ int finish_block(const double* ew, double* cum, int n, const SampleParams& p, double u01,
                                         double* s_w, int* s_first) {
    block_inclusive_scan(ew, cum, n, s_w);
    if (p.min_p > 0.0) {
        const double floor_e = p.min_p * ew[0];
        n = max(1, block_first(ew, n, [&](double e) { return !(e >= floor_e); }, s_first));
    }
    if (p.top_p < 1.0) {
        const double want = p.top_p * cum[n - 1];
        n = min(n, 1 + block_first(cum, n, [&](double c) { return c >= want; }, s_first));
    }
    const double u = u01 * cum[n - 1];
    return min(n - 1, block_first(cum, n, [&](double c) { return u < c; }, s_first));
}

// Visits this warp's ntok tokens (from `base`) in token order with the
// visitor f(t, k, q): q (0..4) consecutive tokens t .. t+q-1 per lane, lanes
// in token order, keys k[0..q).  With 16-byte aligned rows whose length is a
// multiple of 4 each lane loads float4/int4 groups, the next group's loads
// issued before this one is visited; otherwise one token per lane.  The
// loops are not unrolled: this code runs once per launch, so its size (the
// instruction fetches) costs more than the loop overhead.  f is called by
// all 32 lanes together.
template <typename F>
Q3_DEV void visit_tokens(const float* z, const int32_t* cnt, int base, int ntok, bool vec, const SampleParams& p,
                         F f) {
    const int lane = threadIdx.x & 31;
    if (vec) {
        const float4* z4 = reinterpret_cast<const float4*>(z + base);
        const int4* c4 = reinterpret_cast<const int4*>(cnt + base);
        float4 zn = make_float4(0.f, 0.f, 0.f, 0.f);
        int4 cn = make_int4(0, 0, 0, 0);
        if (4 * lane < ntok) zn = __ldg(z4 + lane), cn = c4[lane];
#pragma unroll 1
        for (int t0 = 0; t0 < ntok; t0 += 128) {
            const int t = t0 + 4 * lane;
            const float4 zv = zn;
            const int4 cv = cn;
            if (t + 128 < ntok) zn = __ldg(z4 + (t + 128) / 4), cn = c4[(t + 128) / 4];
            uint64_t k[4];
            k[0] = token_key(zv.x, cv.x, p), k[1] = token_key(zv.y, cv.y, p);
            k[2] = token_key(zv.z, cv.z, p), k[3] = token_key(zv.w, cv.w, p);
            f(base + t, k, t < ntok ? 4 : 0);
        }
    } else {
#pragma unroll 1
        for (int t0 = 0; t0 < ntok; t0 += 32) {
            const int t = t0 + lane;
            uint64_t k[4] = {0ull, 0ull, 0ull, 0ull};
            if (t < ntok) k[0] = token_key(__ldg(z + base + t), cnt[base + t], p);
            f(base + t, k, t < ntok ? 1 : 0);
        }
    }
}

__global__ void __cluster_dims__(kSampleCtas, 1, 1) __launch_bounds__(kThreads, 1)
    sample_kernel(const SampleArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SampleSmem& s = *reinterpret_cast<SampleSmem*>(smem_raw);
    cg::cluster_group cl = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)cl.block_rank();
    const int b = blockIdx.x / kSampleCtas;
    const SampleParams p = *a.params;
    const int V = a.V;
    const float* z = a.logits + (size_t)b * a.ldz;
    int32_t* cnt = a.counts + (size_t)b * V;
    const bool vec = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(cnt)) & 15) == 0;
    const int chunk = band_chunk(V), span = chunk / kWarps;
    const int base = rank * chunk + warp * span;     // this warp's first token
    const int ntok = max(0, min(span, V - base));    // and how many it has
    const size_t band_stride = (size_t)kSampleCtas * chunk;
    uint64_t* bkey = a.band_key + (size_t)b * band_stride + base;
    int32_t* btok = a.band_tok + (size_t)b * band_stride + base;
    const int k = min(p.top_k, V);

    for (int i = tid; i < kBins; i += kThreads) s.hist[0][i] = 0;
    if (tid == 0) s.n_sel = 0, s.n_sub = 0;
    __syncthreads();

    // round 0: the top 12 bits of every token's key
    visit_tokens(z, cnt, base, ntok, vec, p, [&](int, const uint64_t* kk, int q) {
        for (int e = 0; e < q; ++e) atomicAdd(&s.hist[0][kk[e] >> 52], 1);
    });
    int need = k, count = 0;
    const int d0 = select_digit(s, 0, need, &count, cl);

    // the keys with a top digit of at least d0 (the "band": every candidate
    // is among them) are listed per warp in token order
    int nb = 0;
    visit_tokens(z, cnt, base, ntok, vec, p, [&](int t, const uint64_t* kk, int q) {
        unsigned in[4];
        int below = 0, total = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            in[e] = __ballot_sync(0xffffffffu, e < q && (int)(kk[e] >> 52) >= d0);
            below += __popc(in[e] & lanemask_lt());
            total += __popc(in[e]);
        }
        int at = nb + below;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((in[e] >> lane) & 1u) bkey[at] = kk[e], btok[at] = t + e, ++at;
        nb += total;
    });
    __syncwarp();

    // rounds 1..5 over the band's keys with digit d0: 12, 12, 12, 12 and the
    // last 4 bits (keys of a larger digit never match the prefix); once
    // the keys sharing the digits found so far are at most kSubMax in the
    // cluster, CTA 0 finishes the selection among them itself
    uint64_t K = (uint64_t)d0 << 52;
    int low = 0;  // the bits of K below `low` are not decided (early finish)
    bool early = false;
#pragma unroll 1
    for (int r = 1; r <= 5; ++r) {
        const int shift = r < 5 ? 52 - 12 * r : 0;
        const int hi = r < 5 ? shift + 12 : 4;
        const int dmask = (1 << (hi - shift)) - 1;
        for (int j = lane; j < nb; j += 32) {
            const uint64_t key = bkey[j];
            if ((key >> hi) == (K >> hi)) atomicAdd(&s.hist[r & 1][(int)(key >> shift) & dmask], 1);
        }
        K |= (uint64_t)select_digit(s, r, need, &count, cl) << shift;
        if (count <= kSubMax) {
            early = true, low = shift;
            break;
        }
    }

    if (early) {
        // keys above K's decided bits are taken; the few that share them go
        // to CTA 0, which sorts them and takes the first `need`
        const uint64_t P = K >> low;
        for (int j = lane; j < nb; j += 32) {
            const uint64_t key = bkey[j];
            if ((key >> low) > P) {
                select_one(s, key, btok[j]);
            } else if ((key >> low) == P) {
                const int i = atomicAdd(&s.n_sub, 1);
                if (i < kSubMax) s.sub_key[i] = key, s.sub_tok[i] = btok[j];
            }
        }
        cl.sync();
        if (rank == 0 && warp == 0) {
            int m = min(s.n_sub, kSubMax);
            for (int peer = 1; peer < kSampleCtas; ++peer) {
                const SampleSmem& ps = *cl.map_shared_rank(&s, peer);
                const int pn = min(ps.n_sub, kSubMax);
                for (int i = lane; i < pn && m + i < kSubMax; i += 32)
                    s.sub_key[m + i] = ps.sub_key[i], s.sub_tok[m + i] = ps.sub_tok[i];
                m = min(kSubMax, m + pn);
            }
            __syncwarp();
            bitonic(s.sub_key, s.sub_tok, m, 32, [] { __syncwarp(); });
            for (int i = lane; i < min(need, m); i += 32) select_one(s, s.sub_key[i], s.sub_tok[i]);
        }
        cl.sync();  // the peers keep their lists until CTA 0 has read them
    } else {
        // K is the k-th largest key: every key above it is taken, and of the
        // keys equal to it the `need` with the lowest tokens
        int my_ties = 0;
        for (int j0 = 0; j0 < nb; j0 += 32) {
            const int j = j0 + lane;
            const uint64_t key = j < nb ? bkey[j] : 0ull;
            if (j < nb && key > K) select_one(s, key, btok[j]);
            my_ties += __popc(__ballot_sync(0xffffffffu, j < nb && key == K));
        }
        if (lane == 0) s.tie_before[warp] = my_ties;
        __syncthreads();
        if (tid == 0) {
            int c = 0;
            for (int w = 0; w < kWarps; ++w) {
                const int x = s.tie_before[w];
                s.tie_before[w] = c;
                c += x;
            }
            s.ties = c;
        }
        cl.sync();
        int off = s.tie_before[warp];
        for (int peer = 0; peer < rank; ++peer) off += *cl.map_shared_rank(&s.ties, peer);
        for (int j0 = 0; j0 < nb; j0 += 32) {
            const int j = j0 + lane;
            const bool tie = j < nb && bkey[j] == K;
            const unsigned m = __ballot_sync(0xffffffffu, tie);
            if (tie && off + __popc(m & lanemask_lt()) < need) select_one(s, K, btok[j]);
            off += __popc(m);
        }
    }

    // each CTA sorts its candidates; their exponentials, relative to the
    // largest temperature-scaled logit of the cluster, spread over the 8 SMs
    __syncthreads();
    const int mine = min(s.n_sel, kSampleMaxTopK);
    sort_candidates(s.key, s.tok, mine);
    if (tid == 0) s.kmax = mine ? s.key[0] : 0ull;
    cl.sync();
    unsigned long long kmax = 0ull;
    for (int peer = 0; peer < kSampleCtas; ++peer) kmax = max(kmax, *cl.map_shared_rank(&s.kmax, peer));
    const double vmax = __ddiv_rn(key_value(kmax), p.temperature);
    for (int i = tid; i < mine; i += kThreads)
        s.e[i] = exp(__dsub_rn(__ddiv_rn(key_value(s.key[i]), p.temperature), vmax));

    // CTA 0 gathers the peers' sorted runs behind its own
    cl.sync();
    if (rank == 0) {
        if (tid < kSampleCtas) s.run_off[tid + 1] = max(0, tid ? cl.map_shared_rank(&s, tid)->n_sel : s.n_sel);
        __syncthreads();
        if (tid == 0) {
            s.run_off[0] = 0;
            for (int r = 0; r < kSampleCtas; ++r) s.run_off[r + 1] = min(kSampleMaxTopK, s.run_off[r] + s.run_off[r + 1]);
        }
        __syncthreads();
        for (int idx = s.run_off[1] + tid; idx < s.run_off[kSampleCtas]; idx += kThreads) {
            int r = 1;
            while (r < kSampleCtas - 1 && s.run_off[r + 1] <= idx) ++r;
            const SampleSmem& ps = *cl.map_shared_rank(&s, r);
            const int i = idx - s.run_off[r];
            s.key[idx] = ps.key[i], s.tok[idx] = ps.tok[i], s.e[idx] = ps.e[i];
        }
    }
    cl.sync();  // the peers stay resident until CTA 0 has read them
    if (rank != 0) return;
    int n = s.run_off[kSampleCtas];
    if (n != k && tid == 0 && a.status) atomicExch(a.status, kStatusSampleSelect);

    // merge the 8 runs: a candidate's place is its index in its own run plus
    // the candidates of the other runs that come before it (binary search)
    int* mtok = &s.hist[0][0];
    for (int idx = tid; idx < n; idx += kThreads) {
        int r = 0;
        while (r < kSampleCtas - 1 && s.run_off[r + 1] <= idx) ++r;
        const uint64_t kk = s.key[idx];
        const int tt = s.tok[idx];
        int pos = idx - s.run_off[r];
        for (int r2 = 0; r2 < kSampleCtas; ++r2) {
            if (r2 == r) continue;
            int lo = s.run_off[r2], hi = s.run_off[r2 + 1];
            const int start = lo;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (before(s.key[mid], s.tok[mid], kk, tt)) lo = mid + 1;
                else hi = mid;
            }
            pos += lo - start;
        }
        mtok[pos] = tt, s.w[pos] = s.e[idx];
    }
    if (n == 0 && tid == 0) mtok[0] = 0, s.w[0] = 1.0;  // keeps the reads below in range
    n = max(n, 1);
    __syncthreads();

    const int step = a.step ? *a.step - 1 : a.step_value;
    const double u01 = uniform_draw(p.seed, (uint32_t)b, (uint32_t)step);
    int pick;
    if (n <= kSmallN) {
        if (warp != 0) return;
        pick = finish_small(s.w, s.e, n, p, u01);
    } else {
        pick = finish_block(s.w, s.e, n, p, u01, s.dbl, &s.first);
    }
    if (tid == 0) {
        const int token = mtok[pick];
        a.tokens[b] = token;
        if (a.out_ids && step >= 0 && step < a.out_cap) a.out_ids[(size_t)b * a.out_cap + step] = token;
        cnt[token] += 1;
    }
}

__global__ void count_tokens_kernel(const int32_t* ids, const int32_t* row_seq, int M, int32_t* counts, int V) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m < M) {
        const int t = ids[m];
        if (t >= 0 && t < V) atomicAdd(counts + (size_t)row_seq[m] * V + t, 1);
    }
}

}  // namespace

size_t sample_band_entries(int V) { return (size_t)kSampleCtas * band_chunk(V); }

cudaError_t launch_sample(const SampleArgs& a, int B, cudaStream_t st) {
    static_assert(kSampleMaxTopK % kThreads == 0, "scan ownership");
    static_assert(kBins == 4 * kThreads, "histogram ownership");
    if (B < 1) return cudaSuccess;
    cudaError_t e = allow_max_dynamic_smem((const void*)sample_kernel);
    if (e != cudaSuccess) return e;
    sample_kernel<<<B * kSampleCtas, kThreads, sizeof(SampleSmem), st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_count_tokens(const int32_t* ids, const int32_t* row_seq, int M, int32_t* counts, int V,
                                cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    count_tokens_kernel<<<(M + 255) / 256, 256, 0, st>>>(ids, row_seq, M, counts, V);
    return cudaGetLastError();
}

}  // namespace q3
