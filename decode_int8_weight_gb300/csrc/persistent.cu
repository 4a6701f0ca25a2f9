// The decode step as one persistent kernel (sm_103a).
//
// One CTA per SM, launched cooperatively so that every CTA is resident.
// Warp 8 of each CTA is a producer: it walks the CTA's share of the step --
// weight tiles of every projection of every layer, then of the tied lm_head,
// and the KV-cache chunks of its attention work -- and streams them with 1-D
// bulk copies (TMA) into a ring of shared-memory slots, as far ahead as the
// ring allows.  None of those bytes depends on this step's activations, so
// the producer crosses layer and phase boundaries freely and HBM stays busy
// while the consumers wait on data dependencies.
//
// Warps 0-7 consume the ring in the same order.  Per layer the phases are
//   QKV  : int8 GEMV, out = s * r * (W . (g_attn * x))      (r = 1/rms(x))
//   ATT  : per (sequence, kv head) split-KV attention over the cache chunks,
//          with QK-RMSNorm, RoPE and the bf16 KV append of the new position;
//          the last split to finish merges the partial softmax states
//   O    : x += s * (W . o); writes g_ffn * x planes and per-tile sum(x^2)
//   GU   : a = silu(s_g r (Wg . g x)) * (s_u r (Wu . g x))
//   DOWN : x += s * (W . a); writes g_attn' * x planes and per-tile sum(x^2)
// and at the end the lm_head GEMV with a block-then-grid argmax.  RMSNorm is
// folded into the epilogues: the producing phase writes g*x and partial sums
// of squares, the consuming phase applies 1/rms as a per-sequence scalar.
//
// Intermediate values travel between CTAs as 8-byte words {payload, flag}
// written with one 64-bit store; flag is the (step, layer, phase) epoch, so a
// consumer polls the very words it needs and no counters, fences or grid
// barriers sit on the dependency path.  Every wait is bounded; a wait that
// gives up records status 7 and raises an abort flag that ends every wait in
// the grid, and the CTA drains its in-flight copies before returning.
#include "common.cuh"
#include "engine.h"
#include "kernels.h"
#include "persistent.h"

namespace q3 {

constexpr int kSlotBytes = kTileHeader + 16384;  // header + 32 k-pairs of fragments
constexpr int kKpPerChunk = 32;
constexpr int kCWarps = 8;
constexpr int kCThreads = 32 * kCWarps;
constexpr int kThreads = kCThreads + 32;
constexpr int kKvChunk = 64;

// phase ids inside a layer (epoch = base + 8 * layer + phase)
enum { kPhEmbed = 0, kPhQkv = 1, kPhAtt = 2, kPhO = 3, kPhGu = 4, kPhDown = 5 };

Q3_DEV void ll_put(LLw* p, uint32_t payload, uint32_t flag) {
    const unsigned long long v = ((unsigned long long)flag << 32) | payload;
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

Q3_DEV unsigned long long ll_get(const LLw* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

Q3_DEV float ld_cg_f32(const float* p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

struct Shared {
    float red[kCWarps][8][32][2];   // per-warp partial sums of a tile (NT <= 8)
    float scl[16];                  // row scales of the current tile
    float rnorm[kMaxBatch];         // 1/rms per sequence for the current phase
    float sq[kMaxBatch][16];        // x^2 of the current tile's rows
    float gx[kMaxBatch][16];        // gain * x (or silu(gate) * up) of the current tile
    unsigned long long best[kMaxBatch];
    float qs[8][128];               // normed + rotated queries of one kv group
    float kp[128], vp[128];         // bf16-rounded K/V of the new position
    float wm[kCWarps][8], wl[kCWarps][8];
    float wacc[kCWarps][2][128];    // per-warp attention accumulators (GROUP <= 2)
    int pos[kMaxBatch], nchunk[kMaxBatch];
    int flag_last;
    int abort;
    volatile unsigned int issued;   // slots the producer has issued
    volatile int prod_done;
    uint64_t cbar;                  // consumer-group barrier (8 warp arrivals)
};

struct Ctl {
    const PParams* P;
    Shared* sh;
    uint8_t* ring;
    uint64_t* full;
    uint64_t* empty;
    int ns;
    uint32_t used;     // consumer slot counter (per warp, identical sequence)
    uint32_t cphase;   // consumer-barrier phase
    int warp, lane, tid;
    int layer, phase;  // position in the schedule (diagnostics)
};

Q3_DEV bool aborted(const Ctl& c) {
    return c.sh->abort || *reinterpret_cast<volatile int32_t*>(c.P->abort_flag);
}

// Where a wait gave up (first element of the diagnostic record).
enum WaitSite { kSiteFull = 1, kSiteEmpty = 2, kSiteCbar = 3, kSiteWord = 4 };

Q3_DEV uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// A wait gives up after kWaitNs of wall time (checked every 256 polls) or
// kSpinLimit * 16 polls, whichever comes first.
constexpr uint64_t kWaitNs = 2000000000ull;

// Record the first failure of the grid: {site, cta, warp, layer, phase, aux}.
Q3_DEV void raise_abort(Ctl& c, int site, uint32_t aux) {
    c.sh->abort = 1;
    if (atomicCAS(c.P->status, 0, kStatusTimeout) == 0) {
        int32_t* d = c.P->diag;
        d[0] = site, d[1] = blockIdx.x, d[2] = c.warp, d[3] = c.layer, d[4] = c.phase, d[5] = (int32_t)aux;
    }
    atomicExch(c.P->abort_flag, 1);
}

// Shared polling discipline: true when ready() holds, false on abort/timeout.
template <class F>
Q3_DEV bool poll(Ctl& c, int site, uint32_t aux, int sleep_ns, F ready) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (ready()) return true;
        if ((i & 255) == 255) {
            if (aborted(c)) return false;
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitNs || i > kSpinLimit * 16) {
                raise_abort(c, site, aux);
                return false;
            }
        }
        if (i > 16) __nanosleep(sleep_ns);
    }
}

Q3_DEV bool mbar_wait_ctl(Ctl& c, uint64_t* bar, uint32_t parity, int site) {
    return poll(c, site, parity, 32, [&] { return mbar_try_wait(bar, parity); });
}

// all eight consumer warps meet (mbarrier based, so that it can time out)
Q3_DEV bool cbar_sync(Ctl& c) {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.sh->cbar);
    const bool ok = mbar_wait_ctl(c, &c.sh->cbar, c.cphase & 1, kSiteCbar);
    c.cphase++;
    __syncwarp();
    return ok;
}

Q3_DEV bool slot_wait(Ctl& c, uint8_t*& slot) {
    const int s = (int)(c.used % c.ns);
    if (!mbar_wait_ctl(c, &c.full[s], (c.used / c.ns) & 1, kSiteFull)) return false;
    slot = c.ring + (size_t)s * kSlotBytes;
    return true;
}

Q3_DEV void slot_release(Ctl& c) {
    const int s = (int)(c.used % c.ns);
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.empty[s]);
    c.used++;
}

// Re-poll *p until the word already loaded into v carries `flag`.  Callers
// issue all their loads first (ll_get) and settle them afterwards, so the
// L2 round trips of one wait overlap.
Q3_DEV bool ll_settle(Ctl& c, const LLw* p, uint32_t flag, unsigned long long& v) {
    if ((uint32_t)(v >> 32) == flag) return true;
    return poll(c, kSiteWord, flag, 20, [&] {
        v = ll_get(p);
        return (uint32_t)(v >> 32) == flag;
    });
}

// wait until *p carries `flag`; return its payload
Q3_DEV bool ll_wait(Ctl& c, const LLw* p, uint32_t flag, uint32_t& out) {
    unsigned long long v = ll_get(p);
    if (!ll_settle(c, p, flag, v)) return false;
    out = (uint32_t)v;
    return true;
}

// ------------------------------------------------------------------ schedule
// Tile t of a phase instance goes to CTA (t + rot) mod G, rot running over
// the step so that every CTA gets the same share of bytes.
Q3_DEV int first_tile(int cta, int rot, int G) { return ((cta - rot) % G + G) % G; }

// Attention work of a layer: chunk list ordered by (sequence, kv head, chunk),
// CTA i owns chunks [floor(i T / G), floor((i + 1) T / G)).
struct AttnSched {
    int T, G, nkv, B;
    const int* nchunk;  // per sequence
    Q3_DEV long long start(int i) const { return (long long)i * T / G; }
    Q3_DEV int cta_of(long long j) const {
        int i = (int)((j * G) / T);
        while (i > 0 && start(i) > j) --i;
        while (i + 1 < G && start(i + 1) <= j) ++i;
        return i;
    }
    // chunk j -> (b, g, c, first chunk of (b, g))
    Q3_DEV void locate(long long j, int& b, int& g, int& cc, long long& s0) const {
        long long base = 0;
        for (b = 0; b < B; ++b) {
            const long long n = (long long)nkv * nchunk[b];
            if (j < base + n) break;
            base += n;
        }
        const int C = nchunk[b];
        g = (int)((j - base) / C);
        cc = (int)((j - base) % C);
        s0 = base + (long long)g * C;
    }
};

// ------------------------------------------------------------------ producer
__device__ __noinline__ void produce(Ctl& c) {
    const PParams& P = *c.P;
    Shared& sh = *c.sh;
    const int cta = blockIdx.x, G = gridDim.x;
    uint32_t issued = 0;
    bool ok = true;
    auto put = [&](const void* src, uint32_t bytes) {
        if (!ok) return;
        const int s = (int)(issued % c.ns);
        if (issued >= (uint32_t)c.ns) {
            if (!mbar_wait_ctl(c, &c.empty[s], ((issued / c.ns) - 1) & 1, kSiteEmpty)) {
                ok = false;
                return;
            }
        }
        mbar_arrive_expect_tx(&c.full[s], bytes);
        bulk_g2s(c.ring + (size_t)s * kSlotBytes, src, bytes, &c.full[s]);
        issued++;
        sh.issued = issued;
    };
    auto put_tile = [&](const uint8_t* blob, int K) {
        const size_t total = tile_blob_bytes(K);
        size_t off = 0;
        while (off < total && ok) {
            const size_t chunk = off == 0 ? (total < (size_t)kSlotBytes ? total : (size_t)kSlotBytes)
                                          : (total - off < 16384 ? total - off : 16384);
            put(blob + off, (uint32_t)chunk);
            off += chunk;
        }
    };
    auto put_phase = [&](const uint8_t* blobs, int ntiles, int K, int& rot) {
        for (int t = first_tile(cta, rot, G); t < ntiles && ok; t += G) put_tile(blobs + (size_t)t * tile_blob_bytes(K), K);
        rot = (rot + ntiles) % G;
    };
    const int H = P.H, I = P.I, hd = P.hd;
    const int Dq = P.nh * hd;
    int rot = (P.H / 16) % G;  // the embedding phase's tiles come first
    AttnSched as{0, G, P.nkv, P.B, sh.nchunk};
    for (int b = 0; b < P.B; ++b) as.T += P.nkv * sh.nchunk[b];
    const long long a0 = as.start(cta), a1 = as.start(cta + 1);
    const uint32_t kvbytes = (uint32_t)(kKvChunk * hd * 2);
    for (int l = 0; l < P.L && ok; ++l) {
        put_phase(P.mats[4 * l + 0], P.qkv_rows / 16, H, rot);
        for (long long j = a0; j < a1 && ok; ++j) {
            int b, g, cc;
            long long s0;
            as.locate(j, b, g, cc, s0);
            const size_t base = ((((size_t)l * P.bmax + b) * P.nkv + g) * P.cap + (size_t)cc * kKvChunk) * hd;
            put(P.kc + base, kvbytes);
            put(P.vc + base, kvbytes);
        }
        put_phase(P.mats[4 * l + 1], H / 16, Dq, rot);
        put_phase(P.mats[4 * l + 2], 2 * I / 16, H, rot);
        put_phase(P.mats[4 * l + 3], H / 16, I, rot);
    }
    put_phase(P.lm, P.vpad / 16, H, rot);
    sh.prod_done = 1;
}

// ------------------------------------------------------------------ consumer pieces

// 1/rms(x) per sequence from the per-tile partial sums of squares
Q3_DEV bool load_rnorm(Ctl& c, const LLw* ss, uint32_t flag) {
    const PParams& P = *c.P;
    const int ntiles = P.H / 16;
    for (int b = c.warp; b < P.B; b += kCWarps) {
        float acc = 0.f;
        for (int j0 = c.lane; j0 < ntiles; j0 += 128) {
            unsigned long long raw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + 32 * u < ntiles) raw[u] = ll_get(ss + (size_t)(j0 + 32 * u) * P.bmax + b);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + 32 * u < ntiles) {
                    if (!ll_settle(c, ss + (size_t)(j0 + 32 * u) * P.bmax + b, flag, raw[u])) return false;
                    acc += __uint_as_float((uint32_t)raw[u]);
                }
        }
        acc = warp_sum(acc);
        if (c.lane == 0) c.sh->rnorm[b] = 1.0f / sqrtf(acc / (float)P.H + P.eps);
    }
    return cbar_sync(c);
}

// One 16-row weight tile against the activation planes plane[b][k]
// ({f16 hi, f16 lo} of each value); leaves per-warp sums in sh.red and the
// row scales in sh.scl (visible to all consumer threads on return).
template <int NT>
__device__ __noinline__ bool gemv_tile(Ctl& c, int K, const LLw* plane, uint32_t flag) {
    const PParams& P = *c.P;
    const int KP = K >> 5;
    const int nchunks = (KP + kKpPerChunk - 1) / kKpPerChunk;
    const int g = c.lane >> 2, t = c.lane & 3;
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    constexpr int KB = NT == 1 ? 4 : (NT == 2 ? 2 : 1);  // k-pairs whose operands are in flight together
    for (int j = 0; j < nchunks; ++j) {
        uint8_t* slot;
        if (!slot_wait(c, slot)) return false;
        if (j == 0 && c.warp == 0 && c.lane < 16) c.sh->scl[c.lane] = reinterpret_cast<const float*>(slot)[c.lane];
        const uint8_t* fb = slot + (j == 0 ? kTileHeader : 0);
        const int kp_end = min(KP, kKpPerChunk * (j + 1));
        for (int i0 = 0; i0 < 4; i0 += KB) {
            // B operand: the four {v(k), v(k+1)} words of this lane's column
            // (sequence 4n + g/2, hi part for even g, lo part for odd g)
            unsigned long long raw[KB][NT][4];
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int p = kKpPerChunk * j + c.warp + 8 * (i0 + i);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int b = 4 * n + (g >> 1);
                    if (p < kp_end && b < P.B) {
                        const LLw* base = plane + (size_t)(2 * b + (g & 1)) * (K >> 1) + 16 * p + t;
#pragma unroll
                        for (int e = 0; e < 4; ++e) raw[i][n][e] = ll_get(base + 4 * e);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int p = kKpPerChunk * j + c.warp + 8 * (i0 + i);
                if (p >= kp_end) continue;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int b = 4 * n + (g >> 1);
                    if (b < P.B) {
                        const LLw* base = plane + (size_t)(2 * b + (g & 1)) * (K >> 1) + 16 * p + t;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (!ll_settle(c, base + 4 * e, flag, raw[i][n][e])) return false;
                    }
                }
                const uint4 wv = *reinterpret_cast<const uint4*>(fb + (size_t)(p - kKpPerChunk * j) * 512 + c.lane * 16);
                uint32_t A0[4], A1[4];
                u8x4_to_f16x2x2(wv.x, A0[0], A0[1]);
                u8x4_to_f16x2x2(wv.y, A0[2], A0[3]);
                u8x4_to_f16x2x2(wv.z, A1[0], A1[1]);
                u8x4_to_f16x2x2(wv.w, A1[2], A1[3]);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const bool live = 4 * n + (g >> 1) < P.B;
                    const uint32_t b0 = live ? (uint32_t)raw[i][n][0] : 0u;
                    const uint32_t b1 = live ? (uint32_t)raw[i][n][1] : 0u;
                    const uint32_t b2 = live ? (uint32_t)raw[i][n][2] : 0u;
                    const uint32_t b3 = live ? (uint32_t)raw[i][n][3] : 0u;
                    mma_f16_16816(acc[n], A0, b0, b1);
                    mma_f16_16816(acc[n], A1, b2, b3);
                }
            }
        }
        slot_release(c);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        c.sh->red[c.warp][n][c.lane][0] = acc[n][0] + acc[n][1];
        c.sh->red[c.warp][n][c.lane][1] = acc[n][2] + acc[n][3];
    }
    return cbar_sync(c);
}

Q3_DEV float red_sum(const Shared& sh, int n, int ln, int half) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) s += sh.red[w][n][ln][half];
    return s;
}

// Activation planes: plane[(2b + part) * (K/2) + k/2] = {v(k), v(k+1)} as
// f16 pairs, part 0 holding the hi parts and part 1 the lo parts -- exactly
// the B-operand registers of the MMA for column (sequence b, part).
Q3_DEV void put_pair(LLw* plane, int K, int b, int k, float v0, float v1, uint32_t f) {
    __half h0, l0, h1, l1;
    split_f16(v0, h0, l0);
    split_f16(v1, h1, l1);
    const uint32_t hi = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
    const uint32_t lo = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    ll_put(plane + (size_t)(2 * b) * (K >> 1) + (k >> 1), hi, f);
    ll_put(plane + (size_t)(2 * b + 1) * (K >> 1) + (k >> 1), lo, f);
}

// Residual epilogue shared by O, DOWN (from GEMV sums) and the embedding
// phase (from the gathered row): x = x_prev + v; writes x and stages
// gain * x and x^2 for finish_rows.
Q3_DEV bool resid_store(Ctl& c, int tile, int row_in_tile, int b, float v, bool add_prev, uint32_t fprev,
                        uint32_t fcur, const float* gain) {
    const PParams& P = *c.P;
    const int row = 16 * tile + row_in_tile;
    float xn = v;
    if (add_prev) {
        uint32_t xp;
        if (!ll_wait(c, P.x + (size_t)b * P.H + row, fprev, xp)) return false;
        xn = __uint_as_float(xp) + v;
    }
    ll_put(P.x + (size_t)b * P.H + row, __float_as_uint(xn), fcur);
    c.sh->gx[b][row_in_tile] = gain[row] * xn;
    c.sh->sq[b][row_in_tile] = xn * xn;
    return true;
}

// After resid_store: publish the planes of gain * x and the tile's sum of x^2.
Q3_DEV bool finish_rows(Ctl& c, int tile, LLw* plane_out, LLw* ss_out, uint32_t fcur) {
    if (!cbar_sync(c)) return false;
    const PParams& P = *c.P;
    if (c.tid < P.B * 8) {
        const int b = c.tid >> 3, j = c.tid & 7;
        put_pair(plane_out, P.H, b, 16 * tile + 2 * j, c.sh->gx[b][2 * j], c.sh->gx[b][2 * j + 1], fcur);
    }
    if (c.tid < P.B) {
        float s = 0.f;
        for (int r = 0; r < 16; ++r) s += c.sh->sq[c.tid][r];
        ll_put(ss_out + (size_t)tile * P.bmax + c.tid, __float_as_uint(s), fcur);
    }
    return true;
}

// ------------------------------------------------------------------ attention segment
// The CTAs first..first+span-1 cover the chunks of (b, g); the ones whose
// chunk range is empty (start(i) == start(i+1)) do not take part, so
// narrive counts the others and the merge skips their slots.
template <int HD, int GROUP>
__device__ __noinline__ bool attn_segment(Ctl& c, const AttnSched& as, int l, int b, int g, int c0, int c1, int first,
                                          int span, int narrive, uint32_t fqkv, uint32_t fatt) {
    const int seg = blockIdx.x - first;
    constexpr int D = HD / 32;
    constexpr int E = HD / 32;
    const PParams& P = *c.P;
    Shared& sh = *c.sh;
    const int p = sh.pos[b];
    const bool has_p = (c1 == sh.nchunk[b]);
    const float* qn = P.gains[4 * l + 2];
    const float* kn = P.gains[4 * l + 3];
    const float2* cs = P.rope + (size_t)p * (HD / 2);
    const size_t head_base = (((size_t)l * P.bmax + b) * P.nkv + g) * P.cap;
    // 1) queries (and the new K / V) of this kv group
    for (int h = c.warp; h < GROUP + (has_p ? 2 : 0); h += kCWarps) {
        int src;
        if (h < GROUP) src = (g * GROUP + h) * HD;
        else if (h == GROUP) src = (P.nh + g) * HD;
        else src = (P.nh + P.nkv + g) * HD;
        float v[E];
        {
            const LLw* qp = P.qkv + (size_t)b * P.qkv_rows + src + c.lane;
            unsigned long long raw[E];
#pragma unroll
            for (int e = 0; e < E; ++e) raw[e] = ll_get(qp + 32 * e);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if (!ll_settle(c, qp + 32 * e, fqkv, raw[e])) return false;
                v[e] = __uint_as_float((uint32_t)raw[e]);
            }
        }
        if (h <= GROUP) {
            const float* gain = h < GROUP ? qn : kn;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss += v[e] * v[e];
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)HD + P.eps);
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], inv), gain[c.lane + 32 * e]);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                const float2 r = cs[c.lane + 32 * e];
                const float a0 = v[e], b0 = v[e + E / 2];
                v[e] = __fsub_rn(__fmul_rn(a0, r.x), __fmul_rn(b0, r.y));
                v[e + E / 2] = __fadd_rn(__fmul_rn(b0, r.x), __fmul_rn(a0, r.y));
            }
        }
        if (h < GROUP) {
#pragma unroll
            for (int e = 0; e < E; ++e) sh.qs[h][c.lane + 32 * e] = v[e];
        } else {
            __nv_bfloat16* dst = (h == GROUP ? P.kc : P.vc) + (head_base + p) * HD;
            float* keep = h == GROUP ? sh.kp : sh.vp;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const __nv_bfloat16 r = __float2bfloat16_rn(v[e]);
                dst[c.lane + 32 * e] = r;
                keep[c.lane + 32 * e] = __bfloat162float(r);
            }
        }
    }
    if (!cbar_sync(c)) return false;
    // 2) online softmax over the cached positions < p of chunks [c0, c1)
    float q[GROUP][D];
#pragma unroll
    for (int h = 0; h < GROUP; ++h)
#pragma unroll
        for (int d = 0; d < D; ++d) q[h][d] = sh.qs[h][c.lane * D + d];
    const float scale = 1.0f / sqrtf((float)HD);
    float m[GROUP], lsum[GROUP], acc[GROUP][D];
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
        m[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) acc[h][d] = 0.f;
    }
    // fold 8 scored positions (-inf = absent) into the running softmax state
    auto absorb = [&](const float (&sc)[GROUP][8], const float (&vv)[8][D]) {
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
            float cm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) cm = fmaxf(cm, sc[h][i]);
            const float mn = fmaxf(m[h], cm);
            if (mn == -INFINITY) continue;
            const float corr = (m[h] == -INFINITY) ? 0.f : expf(m[h] - mn);
            lsum[h] *= corr;
#pragma unroll
            for (int d = 0; d < D; ++d) acc[h][d] *= corr;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float pr = (sc[h][i] == -INFINITY) ? 0.f : expf(sc[h][i] - mn);
                lsum[h] += pr;
#pragma unroll
                for (int d = 0; d < D; ++d) acc[h][d] += pr * vv[i][d];
            }
            m[h] = mn;
        }
    };
    for (int cc = c0; cc < c1; ++cc) {
        uint8_t *ks, *vs;
        if (!slot_wait(c, ks)) return false;
        c.used++;
        const bool okv = slot_wait(c, vs);
        c.used--;
        if (!okv) return false;
        float sc[GROUP][8];
        float vv[8][D];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = c.warp * 8 + i;
            const int pa = cc * kKvChunk + r;
            const __nv_bfloat16* kr = reinterpret_cast<const __nv_bfloat16*>(ks) + (size_t)r * HD + c.lane * D;
            const __nv_bfloat16* vr = reinterpret_cast<const __nv_bfloat16*>(vs) + (size_t)r * HD + c.lane * D;
            float kf[D];
#pragma unroll
            for (int d = 0; d < D; ++d) {
                kf[d] = __bfloat162float(kr[d]);
                vv[i][d] = __bfloat162float(vr[d]);
            }
#pragma unroll
            for (int h = 0; h < GROUP; ++h) {
                float dot = 0.f;
#pragma unroll
                for (int d = 0; d < D; ++d) dot += q[h][d] * kf[d];
                dot = warp_sum(dot);
                sc[h][i] = (pa < p) ? dot * scale : -INFINITY;
            }
        }
        absorb(sc, vv);
        slot_release(c);
        slot_release(c);
    }
    if (has_p && c.warp == 0) {
        float sc[GROUP][8];
        float vv[8][D];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int d = 0; d < D; ++d) vv[i][d] = i == 0 ? sh.vp[c.lane * D + d] : 0.f;
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < D; ++d) dot += q[h][d] * sh.kp[c.lane * D + d];
            sc[h][0] = warp_sum(dot) * scale;
#pragma unroll
            for (int i = 1; i < 8; ++i) sc[h][i] = -INFINITY;
        }
        absorb(sc, vv);
    }
    // 3) merge the eight warps, publish this split's state
    if (c.lane == 0)
        for (int h = 0; h < GROUP; ++h) {
            sh.wm[c.warp][h] = m[h];
            sh.wl[c.warp][h] = lsum[h];
        }
#pragma unroll
    for (int h = 0; h < GROUP; ++h)
#pragma unroll
        for (int d = 0; d < D; ++d) sh.wacc[c.warp][h][c.lane * D + d] = acc[h][d];
    if (!cbar_sync(c)) return false;
    float* part = P.part + (((size_t)b * P.nkv + g) * gridDim.x + seg) * GROUP * (HD + 2);
    for (int i = c.tid; i < GROUP * HD; i += kCThreads) {
        const int h = i / HD, d = i % HD;
        float M = -INFINITY;
        for (int w = 0; w < kCWarps; ++w) M = fmaxf(M, sh.wm[w][h]);
        float L = 0.f, A = 0.f;
        for (int w = 0; w < kCWarps; ++w) {
            if (sh.wm[w][h] == -INFINITY) continue;
            const float f = expf(sh.wm[w][h] - M);
            L += sh.wl[w][h] * f;
            A += sh.wacc[w][h][d] * f;
        }
        part[h * (HD + 2) + d] = A;
        if (d == 0) {
            part[h * (HD + 2) + HD] = M;
            part[h * (HD + 2) + HD + 1] = L;
        }
    }
    __threadfence();
    if (!cbar_sync(c)) return false;
    if (c.tid == 0) {
        const unsigned int old = atomicAdd(P.attn_cnt + ((size_t)l * P.bmax + b) * P.nkv + g, 1u);
        sh.flag_last = (old == (unsigned)(narrive - 1));
    }
    if (!cbar_sync(c)) return false;
    if (sh.flag_last) {
        __threadfence();
        const float* p0 = P.part + (((size_t)b * P.nkv + g) * gridDim.x) * GROUP * (HD + 2);
        for (int i = c.tid; i < GROUP * HD; i += kCThreads) {
            const int h = i / HD, d = i % HD;
            float M = -INFINITY;
            for (int s = 0; s < span; ++s)
                if (as.start(first + s + 1) > as.start(first + s))
                    M = fmaxf(M, ld_cg_f32(p0 + ((size_t)s * GROUP + h) * (HD + 2) + HD));
            float L = 0.f, A = 0.f;
            for (int s = 0; s < span; ++s) {
                if (as.start(first + s + 1) <= as.start(first + s)) continue;
                const float* ps = p0 + ((size_t)s * GROUP + h) * (HD + 2);
                const float ms = ld_cg_f32(ps + HD);
                if (ms == -INFINITY) continue;
                const float f = expf(ms - M);
                L += ld_cg_f32(ps + HD + 1) * f;
                A += ld_cg_f32(ps + d) * f;
            }
            const float o = A / L;
            const float o1 = __shfl_xor_sync(0xffffffffu, o, 1);
            if ((d & 1) == 0) put_pair(P.pl_o, P.nh * HD, b, (g * GROUP + h) * HD + d, o, o1, fatt);
        }
    }
    return cbar_sync(c);
}

// ------------------------------------------------------------------ consumer
template <int NT, int HD, int GROUP>
Q3_DEV void consume(Ctl& c) {
    const PParams& P = *c.P;
    Shared& sh = *c.sh;
    const int cta = blockIdx.x, G = gridDim.x;
    const int H = P.H, I = P.I, B = P.B, Dq = P.nh * HD;
    const uint32_t eb = *reinterpret_cast<volatile uint32_t*>(P.epoch) * 1024u;
    auto ep = [&](int l, int ph) { return eb + 8u * (uint32_t)l + (uint32_t)ph; };
    int rot = 0;

    // embedding gather (phase 0): x = E[tok] * s, planes of g_attn(0) * x
    {
        const int ntiles = H / 16;
        const uint32_t f = ep(0, kPhEmbed);
        for (int t = first_tile(cta, rot, G); t < ntiles; t += G) {
            for (int i = c.tid; i < B * 16; i += kCThreads) {
                const int b = i >> 4, r = i & 15, k = 16 * t + r;
                const int tok = P.tokens[b];
                const float v = (float)P.emb_raw[(size_t)tok * H + k] * P.emb_scale[tok];
                if (!resid_store(c, t, r, b, v, false, 0, f, P.gains[0])) return;
            }
            if (!finish_rows(c, t, P.pl_attn, P.ss_attn, f)) return;
            if (!cbar_sync(c)) return;
        }
        rot = (rot + ntiles) % G;
    }
    AttnSched as{0, G, P.nkv, B, sh.nchunk};
    for (int b = 0; b < B; ++b) as.T += P.nkv * sh.nchunk[b];
    const long long a0 = as.start(cta), a1 = as.start(cta + 1);

    for (int l = 0; l < P.L; ++l) {
        const uint32_t f_in = l == 0 ? ep(0, kPhEmbed) : ep(l - 1, kPhDown);
        c.layer = l;
        // ---- QKV
        c.phase = kPhQkv;
        {
            const int ntiles = P.qkv_rows / 16;
            int t = first_tile(cta, rot, G);
            if (t < ntiles && !load_rnorm(c, P.ss_attn, f_in)) return;
            for (; t < ntiles; t += G) {
                if (!gemv_tile<NT>(c, H, P.pl_attn, f_in)) return;
                for (int i = c.tid; i < NT * 64; i += kCThreads) {
                    const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, b = 4 * n + (ln & 3);
                    if (b >= B) continue;
                    const int rr = (ln >> 2) + 8 * half;
                    const float v = sh.scl[rr] * sh.rnorm[b] * red_sum(sh, n, ln, half);
                    ll_put(P.qkv + (size_t)b * P.qkv_rows + 16 * t + rr, __float_as_uint(v), ep(l, kPhQkv));
                }
                if (!cbar_sync(c)) return;
            }
            rot = (rot + ntiles) % G;
        }
        // ---- attention
        c.phase = kPhAtt;
        for (long long j = a0; j < a1;) {
            int b, g, cc;
            long long s0;
            as.locate(j, b, g, cc, s0);
            const long long seg_end = s0 + sh.nchunk[b] < a1 ? s0 + sh.nchunk[b] : a1;
            const int first = as.cta_of(s0), last = as.cta_of(s0 + sh.nchunk[b] - 1);
            int narrive = 0;
            for (int i = first; i <= last; ++i) narrive += as.start(i + 1) > as.start(i);
            const int c1 = cc + (int)(seg_end - j);
            if (!attn_segment<HD, GROUP>(c, as, l, b, g, cc, c1, first, last - first + 1, narrive, ep(l, kPhQkv),
                                         ep(l, kPhAtt)))
                return;
            j = seg_end;
        }
        // ---- O projection + residual
        c.phase = kPhO;
        {
            const int ntiles = H / 16;
            const uint32_t fprev = l == 0 ? ep(0, kPhEmbed) : ep(l - 1, kPhDown);
            for (int t = first_tile(cta, rot, G); t < ntiles; t += G) {
                if (!gemv_tile<NT>(c, Dq, P.pl_o, ep(l, kPhAtt))) return;
                for (int i = c.tid; i < NT * 64; i += kCThreads) {
                    const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, b = 4 * n + (ln & 3);
                    if (b >= B) continue;
                    const int rr = (ln >> 2) + 8 * half;
                    const float v = sh.scl[rr] * red_sum(sh, n, ln, half);
                    if (!resid_store(c, t, rr, b, v, true, fprev, ep(l, kPhO), P.gains[4 * l + 1])) return;
                }
                if (!finish_rows(c, t, P.pl_ffn, P.ss_ffn, ep(l, kPhO))) return;
                if (!cbar_sync(c)) return;
            }
            rot = (rot + ntiles) % G;
        }
        // ---- gate/up + SiLU
        c.phase = kPhGu;
        {
            const int ntiles = 2 * I / 16;
            int t = first_tile(cta, rot, G);
            if (t < ntiles && !load_rnorm(c, P.ss_ffn, ep(l, kPhO))) return;
            for (; t < ntiles; t += G) {
                if (!gemv_tile<NT>(c, H, P.pl_ffn, ep(l, kPhO))) return;
                for (int i = c.tid; i < NT * 32; i += kCThreads) {
                    const int n = i >> 5, ln = i & 31, gg = ln >> 2, b = 4 * n + (ln & 3);
                    if (b >= B) continue;
                    const float gate = sh.scl[gg] * sh.rnorm[b] * red_sum(sh, n, ln, 0);
                    const float up = sh.scl[gg + 8] * sh.rnorm[b] * red_sum(sh, n, ln, 1);
                    sh.gx[b][gg] = (gate / (1.0f + expf(-gate))) * up;
                }
                if (!cbar_sync(c)) return;
                if (c.tid < B * 4) {
                    const int b = c.tid >> 2, jj = c.tid & 3;
                    put_pair(P.pl_a, I, b, 8 * t + 2 * jj, sh.gx[b][2 * jj], sh.gx[b][2 * jj + 1], ep(l, kPhGu));
                }
                if (!cbar_sync(c)) return;
            }
            rot = (rot + ntiles) % G;
        }
        // ---- down + residual
        c.phase = kPhDown;
        {
            const int ntiles = H / 16;
            const float* gnext = l + 1 < P.L ? P.gains[4 * (l + 1)] : P.final_norm;
            for (int t = first_tile(cta, rot, G); t < ntiles; t += G) {
                if (!gemv_tile<NT>(c, I, P.pl_a, ep(l, kPhGu))) return;
                for (int i = c.tid; i < NT * 64; i += kCThreads) {
                    const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, b = 4 * n + (ln & 3);
                    if (b >= B) continue;
                    const int rr = (ln >> 2) + 8 * half;
                    const float v = sh.scl[rr] * red_sum(sh, n, ln, half);
                    if (!resid_store(c, t, rr, b, v, true, ep(l, kPhO), ep(l, kPhDown), gnext)) return;
                }
                if (!finish_rows(c, t, P.pl_attn, P.ss_attn, ep(l, kPhDown))) return;
                if (!cbar_sync(c)) return;
            }
            rot = (rot + ntiles) % G;
        }
    }
    // ---- lm_head + argmax
    c.layer = P.L;
    c.phase = 6;
    {
        const int ntiles = P.vpad / 16;
        const uint32_t f = ep(P.L - 1, kPhDown);
        if (c.tid < kMaxBatch) sh.best[c.tid] = 0ull;
        int t = first_tile(cta, rot, G);
        if (t < ntiles && !load_rnorm(c, P.ss_attn, f)) return;
        if (!cbar_sync(c)) return;
        for (; t < ntiles; t += G) {
            if (!gemv_tile<NT>(c, H, P.pl_attn, f)) return;
            for (int i = c.tid; i < NT * 64; i += kCThreads) {
                const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, b = 4 * n + (ln & 3);
                if (b >= B) continue;
                const int rr = (ln >> 2) + 8 * half, row = 16 * t + rr;
                if (row >= P.vocab) continue;
                const float z = sh.scl[rr] * sh.rnorm[b] * red_sum(sh, n, ln, half);
                if (P.logits) P.logits[(size_t)b * P.vocab + row] = z;
                atomicMax(&sh.best[b], argmax_key(z, (uint32_t)row));
            }
            if (!cbar_sync(c)) return;
        }
        if (c.tid < B) atomicMax(&P.keys[c.tid], sh.best[c.tid]);
        __threadfence();
        if (!cbar_sync(c)) return;
        if (c.tid == 0) sh.flag_last = (atomicAdd(P.exit_cnt, 1u) == (unsigned)(G - 1));
        if (!cbar_sync(c)) return;
        if (sh.flag_last) {
            __threadfence();
            const int step = *reinterpret_cast<volatile int32_t*>(P.step);
            if (c.tid < B) {
                const int b = c.tid;
                const unsigned long long k = atomicExch(&P.keys[b], 0ull);
                const int tok = (int)argmax_key_index(k);
                P.tokens[b] = tok;
                if (step < P.out_cap) P.out_ids[(size_t)b * P.out_cap + step] = tok;
                if (P.advance_pos) P.pos[b] += 1;
            }
            const int ncnt = P.L * P.bmax * P.nkv;
            for (int i = c.tid; i < ncnt; i += kCThreads) P.attn_cnt[i] = 0u;
            if (c.tid == 0) {
                *P.step = step + 1;
                *P.epoch = *P.epoch + 1u;
                *P.exit_cnt = 0u;
            }
        }
    }
}

template <int NT, int HD, int GROUP>
__global__ void __launch_bounds__(kThreads, 1) persistent_step_kernel(PParams P) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ Shared sh;
    __shared__ PParams sP;
    if (threadIdx.x == 0) sP = P;
    const int ns = P.ns;
    Ctl c;
    c.P = &sP;
    c.sh = &sh;
    c.ring = dsm;
    c.full = reinterpret_cast<uint64_t*>(dsm + (size_t)ns * kSlotBytes);
    c.empty = c.full + ns;
    c.ns = ns;
    c.used = 0;
    c.cphase = 0;
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    c.tid = threadIdx.x;
    c.layer = -1;
    c.phase = -1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], kCWarps);
        }
        mbar_init(&sh.cbar, kCWarps);
        fence_mbar_init();
        sh.abort = 0;
        sh.issued = 0;
        sh.prod_done = 0;
        sh.flag_last = 0;
    }
    if (threadIdx.x < P.B) {
        const int p = P.pos[threadIdx.x];
        sh.pos[threadIdx.x] = p;
        sh.nchunk[threadIdx.x] = p / kKvChunk + 1;
    }
    __syncthreads();
    if (c.warp == kCWarps) {
        if (c.lane == 0) produce(c);
        return;
    }
    consume<NT, HD, GROUP>(c);
    if (sh.abort && c.tid == 0) {
        // give every copy still in flight a bounded chance to land
        for (uint32_t i = 0; i < kSpinLimit && !sh.prod_done; ++i) __nanosleep(64);
        const uint32_t issued = sh.issued;
        for (uint32_t u = c.used; u < issued; ++u) mbar_wait_bounded(&c.full[u % ns], (u / ns) & 1);
        (void)global_ns;
    }
}

// ------------------------------------------------------------------ host side
template <int NT, int HD, int GROUP>
static cudaError_t launch_t(const PParams& P, int grid, size_t smem, cudaStream_t st) {
    auto kern = persistent_step_kernel<NT, HD, GROUP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int HD, int GROUP>
static cudaError_t launch_hg(const PParams& P, int grid, size_t smem, cudaStream_t st) {
    const int nt = (P.B + 3) / 4;
    if (nt <= 1) return launch_t<1, HD, GROUP>(P, grid, smem, st);
    if (nt <= 2) return launch_t<2, HD, GROUP>(P, grid, smem, st);
    if (nt <= 4) return launch_t<4, HD, GROUP>(P, grid, smem, st);
    return launch_t<8, HD, GROUP>(P, grid, smem, st);
}

bool persistent_supported(const q3i8_dims& d) {
    const int group = d.n_heads / d.n_kv_heads;
    return (d.head_dim == 128 || d.head_dim == 64) && group == 2 && d.n_layers <= 127;
}

size_t persistent_static_smem() { return sizeof(Shared); }

int persistent_slots(int max_optin_smem) {
    const int avail = max_optin_smem - (int)sizeof(Shared) - 1024;
    int ns = avail / (kSlotBytes + 16);
    return ns > 12 ? 12 : ns;
}

size_t persistent_dyn_smem(int ns) { return (size_t)ns * kSlotBytes + 2 * (size_t)ns * sizeof(uint64_t); }

cudaError_t launch_persistent_step(const PParams& P, int grid, cudaStream_t st) {
    const size_t smem = persistent_dyn_smem(P.ns);
    if (P.hd == 128) return launch_hg<128, 2>(P, grid, smem, st);
    return launch_hg<64, 2>(P, grid, smem, st);
}

}  // namespace q3
