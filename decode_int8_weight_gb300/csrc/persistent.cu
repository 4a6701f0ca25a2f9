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
// consumer checks the very words it reads and no counters, fences or grid
// barriers sit on the dependency path.  For B <= 4 a CTA copies a phase's
// whole input vector into shared memory once (after one warp has sampled a
// few words of it), and every tile of the phase reads its MMA operands from
// there.  Every wait is bounded; a wait that gives up records where, raises
// status 7 and an abort flag that ends every wait in the grid, and the CTA
// drains its in-flight copies before returning.
#include "common.cuh"
#include "engine.h"
#include "kernels.h"
#include "persistent.h"

namespace q3 {

constexpr int kSlotBytes = kTileHeader + 16384;  // header + 32 k-pairs of fragments
constexpr int kKpPerChunk = 32;
constexpr int kCWarps = 4;
constexpr int kCThreads = 32 * kCWarps;
constexpr int kThreads = kCThreads + 32;
constexpr int kKvChunk = 64;
constexpr int kStagePad = 4;  // u32 padding per staged column (bank spread)
constexpr int kMaxSlots = 12;
constexpr int kMaxHTiles = 4;  // H-row tiles per CTA (H <= 64 * grid)

// phase ids inside a layer (epoch = base + 8 * layer + phase)
enum { kPhEmbed = 0, kPhQkv = 1, kPhAtt = 2, kPhO = 3, kPhGu = 4, kPhDown = 5, kPhLm = 6 };

Q3_DEV void ll_put(LLw* p, uint32_t payload, uint32_t flag) {
    const unsigned long long v = ((unsigned long long)flag << 32) | payload;
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

Q3_DEV unsigned long long ll_get(const LLw* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// two adjacent words (16-byte aligned); each word is checked on its own
Q3_DEV void ll_get2(const LLw* p, unsigned long long& a, unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

Q3_DEV float ld_cg_f32(const float* p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

Q3_DEV void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

struct Shared {
    float scl[16];                  // row scales of the current tile
    float rnorm[kMaxBatch];         // 1/rms per sequence for the current phase
    float sq[kMaxBatch][16];        // x^2 of the current tile's rows
    float gx[kMaxBatch][16];        // gain * x (or silu(gate) * up) of the current tile
    float xres[kMaxHTiles][16][kMaxBatch];  // residual rows of this CTA's H-row tiles
    float ssp[4 * 256];                     // per-tile sums of squares, B <= 4, H <= 4096 (staged path)
    float xsum[kMaxBatch];                  // sum of the staged operand values per sequence (bias correction)
    float xsum_w[kCWarps][4];
    unsigned long long best[kMaxBatch];
    float qs[2][128];               // normed + rotated queries of one kv group (GROUP <= 2)
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
    float* red;        // [8 warps][NT][32][2] partial sums of a tile
    uint32_t* stage;   // [2B][stage_ld] staged f16-pair words of the phase input (NT == 1)
    int stage_ld;
    int ns;
    uint32_t used;     // consumer slot counter (per warp, identical sequence)
    uint32_t cphase;   // consumer-barrier phase
    int warp, lane, tid;
    int layer, phase;  // position in the schedule (diagnostics)
    int dcount;        // detail stamps recorded so far
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

// Slow paths of every wait, out of line so that each call site costs a test
// and a call; they take scalars only, so that the caller's control block
// stays in registers.  `diag` packs (warp, layer, phase) for the record.
struct WaitCtx {
    const PParams* P;
    int* sh_abort;
    int diag;  // warp | layer << 8 | (phase + 1) << 16
};

Q3_DEV bool aborted_w(const WaitCtx& w) {
    return *reinterpret_cast<volatile int*>(w.sh_abort) || *reinterpret_cast<volatile int32_t*>(w.P->abort_flag);
}

Q3_DEV void raise_abort_w(const WaitCtx& w, int site, uint32_t aux) {
    *w.sh_abort = 1;
    if (atomicCAS(w.P->status, 0, kStatusTimeout) == 0) {
        int32_t* d = w.P->diag;
        d[0] = site, d[1] = blockIdx.x, d[2] = w.diag & 255, d[3] = (w.diag >> 8) & 255, d[4] = (w.diag >> 16) - 1;
        d[5] = (int32_t)aux;
    }
    atomicExch(w.P->abort_flag, 1);
}

__device__ __noinline__ bool poll_mbar(const PParams* P, int* sh_abort, int diag, uint64_t* bar, uint32_t parity,
                                       int site) {
    const WaitCtx w{P, sh_abort, diag};
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255) {
            if (aborted_w(w)) return false;
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitNs || i > kSpinLimit * 16) {
                raise_abort_w(w, site, parity);
                return false;
            }
        }
        if (i > 16) __nanosleep(32);
    }
}

__device__ __noinline__ unsigned long long poll_word(const PParams* P, int* sh_abort, int diag, const LLw* p,
                                                     uint32_t flag) {
    const WaitCtx w{P, sh_abort, diag};
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const unsigned long long v = ll_get(p);
        if ((uint32_t)(v >> 32) == flag) return v;
        if ((i & 255) == 255) {
            if (aborted_w(w)) return 0ull;
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitNs || i > kSpinLimit * 16) {
                raise_abort_w(w, kSiteWord, flag);
                return 0ull;
            }
        }
        if (i > 4) __nanosleep(20);
    }
}

// One round of a batched poll found words still stale: sleep briefly and,
// every 64 rounds, check the abort flag and the time limit.  Returns the
// updated start time, or ~0 when the wait has to give up.
__device__ __noinline__ uint64_t poll_tick(const PParams* P, int* sh_abort, int diag, uint32_t i, uint64_t t0,
                                           uint32_t flag) {
    const WaitCtx w{P, sh_abort, diag};
    if ((i & 63) == 63) {
        if (aborted_w(w)) return ~0ull;
        const uint64_t now = global_ns();
        if (t0 == 0) return now;
        if (now - t0 > kWaitNs || i > kSpinLimit * 16) {
            raise_abort_w(w, kSiteWord, flag);
            return ~0ull;
        }
    }
    if (i > 2) __nanosleep(20);
    return t0;
}

Q3_DEV int diag_of(const Ctl& c) { return c.warp | (c.layer & 255) << 8 | (c.phase + 1) << 16; }

Q3_DEV bool mbar_wait_ctl(Ctl& c, uint64_t* bar, uint32_t parity, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    return poll_mbar(c.P, &c.sh->abort, diag_of(c), bar, parity, site);
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

// Ring slot number u (all consumer warps count slots identically).
Q3_DEV bool slot_wait_at(Ctl& c, uint32_t u, uint8_t*& slot) {
    const int s = (int)(u % c.ns);
    if (!mbar_wait_ctl(c, &c.full[s], (u / c.ns) & 1, kSiteFull)) return false;
    slot = c.ring + (size_t)s * kSlotBytes;
    return true;
}

Q3_DEV bool slot_wait(Ctl& c, uint8_t*& slot) { return slot_wait_at(c, c.used, slot); }

Q3_DEV void slot_release(Ctl& c) {
    const int s = (int)(c.used % c.ns);
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.empty[s]);
    c.used++;
}

// Re-poll *p until the word already loaded into v carries `flag`.  Callers
// issue all their loads first and settle them afterwards, so the L2 round
// trips of one wait overlap.
Q3_DEV bool ll_settle(Ctl& c, const LLw* p, uint32_t flag, unsigned long long& v) {
    if ((uint32_t)(v >> 32) == flag) return true;
    v = poll_word(c.P, &c.sh->abort, diag_of(c), p, flag);
    return (uint32_t)(v >> 32) == flag;
}

// wait until *p carries `flag`; return its payload
Q3_DEV bool ll_wait(Ctl& c, const LLw* p, uint32_t flag, uint32_t& out) {
    unsigned long long v = ll_get(p);
    if (!ll_settle(c, p, flag, v)) return false;
    out = (uint32_t)v;
    return true;
}

Q3_DEV void stamp(const Ctl& c, int idx) {
    if (c.P->trace && (c.warp == kCWarps || c.tid == 0))
        c.P->trace[(size_t)blockIdx.x * trace_stride(c.P->L) + idx] = global_ns();
}

// detail stamp inside the traced layer (consumer thread 0 only)
Q3_DEV void dstamp(Ctl& c, int event) {
    if (!c.P->trace || c.layer != kTraceDetailLayer) return;
    if (c.tid == 0 && c.dcount < 32) {
        unsigned long long* t = c.P->trace + (size_t)blockIdx.x * trace_stride(c.P->L) + trace_detail_base(c.P->L);
        t[2 * c.dcount] = clock64();
        t[2 * c.dcount + 1] = (unsigned long long)(16 * c.phase + event);
    }
    c.dcount++;
}

// ------------------------------------------------------------------ schedule
// Tile t of a phase instance goes to CTA (t + rot) mod G, rot running over
// the step so that every CTA gets the same share of bytes.
Q3_DEV int first_tile(int cta, int rot, int G) { return ((cta - rot) % G + G) % G; }

// Attention work of a layer: units (sequence b, kv head g, split) in that
// order, each covering up to Q consecutive 64-position chunks of b's cache;
// Q = max(4, ceil(T / G)) with T the total chunk count, so short contexts
// take one unit per (b, g) and long ones split evenly over the grid.  Unit u
// goes to CTA u mod G.  Splits of one (b, g) merge their softmax states.
struct AttnSched {
    int B, nkv, G, Q, U;
    const int* nchunk;  // per sequence
    Q3_DEV void init(int B_, int nkv_, int G_, const int* nch) {
        B = B_, nkv = nkv_, G = G_, nchunk = nch;
        long long T = 0;
        for (int b = 0; b < B; ++b) T += (long long)nkv * nchunk[b];
        Q = (int)((T + G - 1) / G);
        if (Q < 4) Q = 4;
        U = 0;
        for (int b = 0; b < B; ++b) U += nkv * nsplit(b);
    }
    Q3_DEV int nsplit(int b) const { return (nchunk[b] + Q - 1) / Q; }
    Q3_DEV void locate(int u, int& b, int& g, int& split) const {
        int base = 0;
        for (b = 0; b < B; ++b) {
            const int n = nkv * nsplit(b);
            if (u < base + n) break;
            base += n;
        }
        const int ns = nsplit(b);
        g = (u - base) / ns;
        split = (u - base) % ns;
    }
};

// ------------------------------------------------------------------ producer
Q3_DEV void produce(Ctl& c) {
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
    // QKV, gate/up and lm_head tiles rotate over the grid starting after the
    // CTAs that own the H-row tiles (embedding, O, down)
    int rot = (P.H / 16) % G;
    AttnSched as;
    as.init(P.B, P.nkv, G, sh.nchunk);
    const uint32_t kvbytes = (uint32_t)(kKvChunk * hd * 2);
    for (int l = 0; l < P.L && ok; ++l) {
        put_phase(P.mats[4 * l + 0], P.qkv_rows / 16, H, rot);
        for (int u = cta; u < as.U && ok; u += G) {
            int b, g, split;
            as.locate(u, b, g, split);
            const int c0 = split * as.Q, c1 = min(sh.nchunk[b], c0 + as.Q);
            for (int cc = c0; cc < c1 && ok; ++cc) {
                const size_t base = ((((size_t)l * P.bmax + b) * P.nkv + g) * P.cap + (size_t)cc * kKvChunk) * hd;
                put(P.kc + base, kvbytes);
                put(P.vc + base, kvbytes);
            }
        }
        int fixed = 0;  // O and down: H-row tile t always on CTA t mod G
        put_phase(P.mats[4 * l + 1], H / 16, Dq, fixed);
        put_phase(P.mats[4 * l + 2], 2 * I / 16, H, rot);
        fixed = 0;
        put_phase(P.mats[4 * l + 3], H / 16, I, fixed);
        stamp(c, 2 + 6 * l + 5);
    }
    put_phase(P.lm, P.vpad / 16, H, rot);
    sh.prod_done = 1;
}

// ------------------------------------------------------------------ consumer pieces

// 1/rms(x) per sequence from the per-tile partial sums of squares
Q3_DEV bool rnorm_from(Ctl& c, const LLw* ss, uint32_t flag) {
    const PParams& P = *c.P;
    const int ntiles = P.H / 16;
    for (int b = c.warp; b < P.B; b += kCWarps) {
        float acc = 0.f;
        for (int j0 = c.lane; j0 < ntiles; j0 += 128) {
            unsigned long long raw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                raw[u] = j0 + 32 * u < ntiles ? ll_get(ss + (size_t)(j0 + 32 * u) * P.bmax + b)
                                              : (unsigned long long)flag << 32;
            uint64_t t0 = 0;
            for (uint32_t i = 0;; ++i) {
                bool stale = false;
#pragma unroll
                for (int u = 0; u < 4; ++u) stale |= (uint32_t)(raw[u] >> 32) != flag;
                if (!stale) break;
                t0 = poll_tick(c.P, &c.sh->abort, diag_of(c), i, t0, flag);
                if (t0 == ~0ull) return false;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if ((uint32_t)(raw[u] >> 32) != flag) raw[u] = ll_get(ss + (size_t)(j0 + 32 * u) * P.bmax + b);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + 32 * u < ntiles) acc += __uint_as_float((uint32_t)raw[u]);
        }
        acc = warp_sum(acc);
        if (c.lane == 0) c.sh->rnorm[b] = 1.0f / sqrtf(acc / (float)P.H + P.eps);
    }
    return true;
}

Q3_DEV bool load_rnorm(Ctl& c, const LLw* ss, uint32_t flag) {
    if (!rnorm_from(c, ss, flag)) return false;
    return cbar_sync(c);
}

// Copy the phase input (plane words of 2B columns x K/2 pairs) into shared
// memory as plain f16 pairs, and 1/rms per sequence when ss is given.  All
// loads of a batch -- plane words and the partial sums of squares -- are
// issued before any is checked, so a stage costs one round trip when its
// input is ready.
Q3_DEV bool stage_plane(Ctl& c, const LLw* plane, int K, uint32_t flag, const LLw* ss, uint32_t sflag) {
    const PParams& P = *c.P;
    const int half = K >> 1;
    const int npair = P.B * half;  // (hi word, lo word) pairs are not adjacent; load word pairs of one part
    const int nss = ss ? P.B * (P.H / 16) : 0;
    // sums of squares: thread i < nss loads word (j = i / B, b = i % B)
    unsigned long long sv = 0;
    if (c.tid < nss) sv = ll_get(ss + (size_t)(c.tid / P.B) * P.bmax + c.tid % P.B);
    constexpr int U = 12;
    float xs[4] = {0.f, 0.f, 0.f, 0.f};  // B <= 4 on this path
    const unsigned long long done = (unsigned long long)flag << 32;
    for (int base = c.tid; base < npair; base += kCThreads * U) {
        unsigned long long v[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = base + u * kCThreads;
            if (q < npair) ll_get2(plane + 2 * q, v[u][0], v[u][1]);
            else v[u][0] = v[u][1] = done;
        }
        // words still stale are re-read together, so a round costs one
        // round trip however many of them were early; this thread's sum of
        // squares word (first batch) rides along
        const bool own_ss = base == c.tid && c.tid < nss;
        uint64_t t0 = 0;
        for (uint32_t i = 0;; ++i) {
            bool stale = own_ss && (uint32_t)(sv >> 32) != sflag;
#pragma unroll
            for (int u = 0; u < U; ++u)
                stale |= ((uint32_t)(v[u][0] >> 32) != flag) | ((uint32_t)(v[u][1] >> 32) != flag);
            if (!stale) break;
            t0 = poll_tick(c.P, &c.sh->abort, diag_of(c), i, t0, flag);
            if (t0 == ~0ull) return false;
            if (own_ss && (uint32_t)(sv >> 32) != sflag) sv = ll_get(ss + (size_t)(c.tid / P.B) * P.bmax + c.tid % P.B);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = base + u * kCThreads;
                if (((uint32_t)(v[u][0] >> 32) != flag) | ((uint32_t)(v[u][1] >> 32) != flag))
                    ll_get2(plane + 2 * q, v[u][0], v[u][1]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = base + u * kCThreads;
            if (q >= npair) continue;
            const int w0 = 2 * q;
            const int col = w0 / half, k2 = w0 - col * half;
            uint32_t* d = c.stage + (size_t)col * c.stage_ld + k2;
            d[0] = (uint32_t)v[u][0];
            d[1] = (uint32_t)v[u][1];
            const __half2 h0 = *reinterpret_cast<const __half2*>(&d[0]);
            const __half2 h1 = *reinterpret_cast<const __half2*>(&d[1]);
            const float part = (__low2float(h0) + __high2float(h0)) + (__low2float(h1) + __high2float(h1));
            const int bb = col >> 1;
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2)
                if (q2 == bb) xs[q2] += part;
        }
    }
    // per-sequence sums of the operand values (hi + lo), fixed order
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
        const float w = warp_sum(xs[q2]);
        if (c.lane == 0) c.sh->xsum_w[c.warp][q2] = w;
    }
    if (ss) {
        // each sequence's H/16 partial sums, in a fixed order: thread-local
        // words go through shared memory and thread b < B adds them up
        float* part = c.sh->ssp;
        if (c.tid < nss) {
            if (!ll_settle(c, ss + (size_t)(c.tid / P.B) * P.bmax + c.tid % P.B, sflag, sv)) return false;
            part[c.tid] = __uint_as_float((uint32_t)sv);
        }
        for (int i = c.tid + kCThreads; i < nss; i += kCThreads) {
            uint32_t u32;
            if (!ll_wait(c, ss + (size_t)(i / P.B) * P.bmax + i % P.B, sflag, u32)) return false;
            part[i] = __uint_as_float(u32);
        }
        if (!cbar_sync(c)) return false;
        if (c.tid < P.B) {
            float acc = 0.f;
            for (int j = 0; j < P.H / 16; ++j) acc += part[j * P.B + c.tid];
            c.sh->rnorm[c.tid] = 1.0f / sqrtf(acc / (float)P.H + P.eps);
        }
    } else {
        if (!cbar_sync(c)) return false;
    }
    if (c.tid < P.B) {
        float t4 = 0.f;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) t4 += c.sh->xsum_w[w][c.tid];
        c.sh->xsum[c.tid] = kBias * t4;
    }
    return cbar_sync(c);
}

// One 16-row weight tile against the activation planes ({f16 hi, f16 lo}
// pairs of each value); split-K over the eight warps.  Leaves per-warp sums
// in c.red and the row scales in sh.scl (visible to all consumer threads on
// return).  NT == 1 reads the operands from the staged copy in shared
// memory, larger NT straight from the flagged words in global memory.
template <int NT>
Q3_DEV bool gemv_tile(Ctl& c, int K, const LLw* plane, uint32_t flag) {
    const PParams& P = *c.P;
    const int KP = K >> 5;
    const int nchunks = (KP + kKpPerChunk - 1) / kKpPerChunk;
    const int g = c.lane >> 2, t = c.lane & 3;
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    dstamp(c, 8);
    for (int j = 0; j < nchunks; ++j) {
        uint8_t* slot;
        if (!slot_wait(c, slot)) return false;
        dstamp(c, 4);
        if (j == 0 && c.warp == 0 && c.lane < 16) c.sh->scl[c.lane] = reinterpret_cast<const float*>(slot)[c.lane];
        const uint8_t* fb = slot + (j == 0 ? kTileHeader : 0);
        const int kp_end = min(KP, kKpPerChunk * (j + 1));
        if constexpr (NT == 1) {
            const bool live = (g >> 1) < P.B;
            const uint32_t sca = smem_u32(c.stage + (size_t)g * c.stage_ld + t);
            const uint32_t fa = smem_u32(fb) + c.lane * 16;
            float a4[4][4];
#pragma unroll
            for (int q = 0; q < 4; ++q) a4[q][0] = a4[q][1] = a4[q][2] = a4[q][3] = 0.f;
            // every operand of this warp's k-pairs is loaded before the first
            // MMA, so the shared-memory latency is paid once per slot
            constexpr int NI = kKpPerChunk / kCWarps;
            uint4 wv[NI];
            uint32_t bq[NI][4];
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int p = kKpPerChunk * j + c.warp + kCWarps * i;
                const bool in = p < kp_end;
                const uint32_t ba = sca + 4 * 16 * p;
                wv[i] = in ? lds128(fa + (p - kKpPerChunk * j) * 512) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int e = 0; e < 4; ++e) bq[i][e] = (in && live) ? lds32(ba + 16 * e) : 0u;
            }
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                // a k-pair past the end multiplies zero operands
                uint32_t A0[4], A1[4];
                u8x4_to_biased(wv[i].x, A0[0], A0[1]);
                u8x4_to_biased(wv[i].y, A0[2], A0[3]);
                u8x4_to_biased(wv[i].z, A1[0], A1[1]);
                u8x4_to_biased(wv[i].w, A1[2], A1[3]);
                mma_f16_16816(a4[(2 * i) & 3], A0, bq[i][0], bq[i][1]);
                mma_f16_16816(a4[(2 * i + 1) & 3], A1, bq[i][2], bq[i][3]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[0][e] += (a4[0][e] + a4[1][e]) + (a4[2][e] + a4[3][e]);
        } else {
            constexpr int KB = NT == 2 ? 4 : (NT == 4 ? 2 : 1);  // k-pairs with operands in flight together
            for (int i0 = 0; i0 < kKpPerChunk / kCWarps; i0 += KB) {
                // B operand: the four {v(k), v(k+1)} words of this lane's column
                // (sequence 4n + g/2, hi part for even g, lo part for odd g)
                unsigned long long raw[KB][NT][4];
#pragma unroll
                for (int i = 0; i < KB; ++i) {
                    const int p = kKpPerChunk * j + c.warp + kCWarps * (i0 + i);
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const int b = 4 * n + (g >> 1);
                        const LLw* base = plane + (size_t)(2 * b + (g & 1)) * (K >> 1) + 16 * p + t;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            raw[i][n][e] = (p < kp_end && b < P.B) ? ll_get(base + 4 * e) : (unsigned long long)flag << 32;
                    }
                }
                // stale words are re-read together: one round trip per round
                uint64_t t0 = 0;
                for (uint32_t it = 0;; ++it) {
                    bool stale = false;
#pragma unroll
                    for (int i = 0; i < KB; ++i)
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) stale |= (uint32_t)(raw[i][n][e] >> 32) != flag;
                    if (!stale) break;
                    t0 = poll_tick(c.P, &c.sh->abort, diag_of(c), it, t0, flag);
                    if (t0 == ~0ull) return false;
#pragma unroll
                    for (int i = 0; i < KB; ++i) {
                        const int p = kKpPerChunk * j + c.warp + kCWarps * (i0 + i);
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            const int b = 4 * n + (g >> 1);
                            const LLw* base = plane + (size_t)(2 * b + (g & 1)) * (K >> 1) + 16 * p + t;
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if ((uint32_t)(raw[i][n][e] >> 32) != flag) raw[i][n][e] = ll_get(base + 4 * e);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < KB; ++i) {
                    const int p = kKpPerChunk * j + c.warp + kCWarps * (i0 + i);
                    if (p >= kp_end) continue;
                    const uint4 wv =
                        *reinterpret_cast<const uint4*>(fb + (size_t)(p - kKpPerChunk * j) * 512 + c.lane * 16);
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
        }
        slot_release(c);
        dstamp(c, 5);
    }
    float* red = c.red + (size_t)c.warp * NT * 64;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        red[(n * 32 + c.lane) * 2 + 0] = acc[n][0] + acc[n][1];
        red[(n * 32 + c.lane) * 2 + 1] = acc[n][2] + acc[n][3];
    }
    return cbar_sync(c);
}

// Cross-warp sum of a split-K tile's partial results; with NT == 1 the
// operands were biased (u8x4_to_biased) and the bias term is removed here.
template <int NT>
Q3_DEV float red_sum(const Ctl& c, int n, int ln, int half) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) s += c.red[((size_t)w * NT * 32 + n * 32 + ln) * 2 + half];
    if constexpr (NT == 1) s -= c.sh->xsum[ln & 3];
    return s;
}

// Per-warp tiles for NT == 1 (B <= 4): warp w of the CTA takes every
// kCWarps-th of the CTA's tiles in this phase, runs the whole K with four
// independent MMA accumulator chains and does its own epilogue, so the
// phase needs no CTA barrier.  The slots of the CTA's tile i are
// used + i*nsl ...; each is released by its warp alone (arrival count
// kCWarps) and every warp advances `used` past all of them at the end.
enum WarpMode { kWmQkv = 0, kWmGu = 1, kWmLm = 2 };

Q3_DEV void put_pair(LLw* plane, int K, int b, int k, float v0, float v1, uint32_t f);

Q3_DEV bool warp_tiles(Ctl& c, int mode, int t0, int ntiles, int G, int K, uint32_t fout) {
    const PParams& P = *c.P;
    Shared& sh = *c.sh;
    const int KP = K >> 5, nsl = (KP + kKpPerChunk - 1) / kKpPerChunk;
    const int g = c.lane >> 2, t = c.lane & 3;
    const bool live = (g >> 1) < P.B;
    const uint32_t sca = smem_u32(c.stage + (size_t)g * c.stage_ld + t);  // B operand column of this lane
    int count = 0;
    for (int tile = t0; tile < ntiles; tile += G, ++count) {
        if ((count & (kCWarps - 1)) != c.warp) continue;
        float a[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) a[q][0] = a[q][1] = a[q][2] = a[q][3] = 0.f;
        float s_lo = 0.f, s_hi = 0.f;
        for (int j = 0; j < nsl; ++j) {
            const uint32_t u = c.used + (uint32_t)(count * nsl + j);
            uint8_t* slot;
            if (!slot_wait_at(c, u, slot)) return false;
            const uint32_t sa = smem_u32(slot);
            if (j == 0) {
                s_lo = lds_f32(sa + 4 * g);
                s_hi = lds_f32(sa + 4 * (g + 8));
            }
            const uint32_t fa = sa + (j == 0 ? kTileHeader : 0) + c.lane * 16;
            const int p0 = kKpPerChunk * j, np = min(KP - p0, kKpPerChunk);
            // groups of 8 k-pairs: all operands of a group are loaded before
            // its 16 MMAs (four independent accumulator chains), so the
            // shared-memory latency is paid once per group; k-pairs past the
            // end of the slot multiply zero operands
#pragma unroll 1
            for (int i0 = 0; i0 < np; i0 += 8) {
                uint4 wv[8];
                uint32_t bq[8][4];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const bool in = i0 + i < np;
                    const uint32_t ba = sca + 4 * 16 * (p0 + i0 + i);
                    wv[i] = in ? lds128(fa + (i0 + i) * 512) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) bq[i][e] = (in && live) ? lds32(ba + 16 * e) : 0u;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t A[4];
                    u8x4_to_biased(wv[i].x, A[0], A[1]);
                    u8x4_to_biased(wv[i].y, A[2], A[3]);
                    mma_f16_16816(a[(2 * i) & 3], A, bq[i][0], bq[i][1]);
                    u8x4_to_biased(wv[i].z, A[0], A[1]);
                    u8x4_to_biased(wv[i].w, A[2], A[3]);
                    mma_f16_16816(a[(2 * i + 1) & 3], A, bq[i][2], bq[i][3]);
                }
            }
            __syncwarp();
            if (c.lane == 0) mbar_arrive_cnt(&c.empty[u % c.ns], kCWarps);
        }
        // lane (g, t): rows g and g+8 of the tile for sequence t (hi + lo columns)
        const float bias = t < P.B ? sh.xsum[t] : 0.f;
        const float v0 =
            (((a[0][0] + a[0][1]) + (a[1][0] + a[1][1])) + ((a[2][0] + a[2][1]) + (a[3][0] + a[3][1]))) - bias;
        const float v1 =
            (((a[0][2] + a[0][3]) + (a[1][2] + a[1][3])) + ((a[2][2] + a[2][3]) + (a[3][2] + a[3][3]))) - bias;
        const float r = t < P.B ? sh.rnorm[t] : 0.f;
        if (mode == kWmQkv) {
            if (t < P.B) {
                LLw* dst = P.qkv + (size_t)t * P.qkv_rows + 16 * tile + g;
                ll_put(dst, __float_as_uint(s_lo * r * v0), fout);
                ll_put(dst + 8, __float_as_uint(s_hi * r * v1), fout);
            }
        } else if (mode == kWmGu) {
            // rows g / g+8 are gate / up of unit 8*tile + g; lane + 4 holds unit g + 1
            const float gate = s_lo * r * v0, up = s_hi * r * v1;
            const float act = (gate / (1.0f + expf(-gate))) * up;
            const float nxt = __shfl_down_sync(0xffffffffu, act, 4);
            if (t < P.B && (g & 1) == 0) put_pair(P.pl_a, P.I, t, 8 * tile + g, act, nxt, fout);
        } else {
            if (t < P.B) {
                const int row = 16 * tile + g;
                const float z0 = s_lo * r * v0, z1 = s_hi * r * v1;
                if (row < P.vocab) {
                    if (P.logits) P.logits[(size_t)t * P.vocab + row] = z0;
                    atomicMax(&sh.best[t], argmax_key(z0, (uint32_t)row));
                }
                if (row + 8 < P.vocab) {
                    if (P.logits) P.logits[(size_t)t * P.vocab + row + 8] = z1;
                    atomicMax(&sh.best[t], argmax_key(z1, (uint32_t)(row + 8)));
                }
            }
        }
    }
    c.used += (uint32_t)(count * nsl);
    // the staged input and 1/rms stay in use until every warp is done
    return cbar_sync(c);
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
// phase (from the gathered row).  H-row tile t lives on CTA t mod G in all
// three phases, so the residual rows stay in this CTA's shared memory
// (slot ti = t / G) from the embedding to the last layer: x = x_prev + v;
// stages gain * x and x^2 for finish_rows.
Q3_DEV void resid_store_g(Ctl& c, int tile, int row_in_tile, int b, float v, bool add_prev, float gain) {
    float& xr = c.sh->xres[tile / gridDim.x][row_in_tile][b];
    const float xn = add_prev ? xr + v : v;
    xr = xn;
    c.sh->gx[b][row_in_tile] = gain * xn;
    c.sh->sq[b][row_in_tile] = xn * xn;
}

Q3_DEV void resid_store(Ctl& c, int tile, int row_in_tile, int b, float v, bool add_prev, const float* gain) {
    resid_store_g(c, tile, row_in_tile, b, v, add_prev, gain[16 * tile + row_in_tile]);
}

// After resid_store: publish the planes of gain * x and the tile's sum of x^2.
Q3_DEV bool finish_rows(Ctl& c, int tile, LLw* plane_out, LLw* ss_out, uint32_t fcur) {
    dstamp(c, 6);
    if (!cbar_sync(c)) return false;
    dstamp(c, 7);
    const PParams& P = *c.P;
    for (int i = c.tid; i < P.B * 8; i += kCThreads) {
        const int b = i >> 3, j = i & 7;
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
// One attention unit: chunks [c0, c1) of (b, g), split `split` of nsplit.
template <int HD, int GROUP>
Q3_DEV bool attn_segment(Ctl& c, int l, int b, int g, int c0, int c1, int split, int nsplit,
                                          uint32_t fqkv, uint32_t fatt) {
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
        // gains and rotation of this head, fetched along with its words
        float gn[E];
        float2 rp[E / 2];
        if (h <= GROUP) {
            const float* gain = h < GROUP ? qn : kn;
#pragma unroll
            for (int e = 0; e < E; ++e) gn[e] = gain[c.lane + 32 * e];
#pragma unroll
            for (int e = 0; e < E / 2; ++e) rp[e] = cs[c.lane + 32 * e];
        }
        {
            const LLw* qp = P.qkv + (size_t)b * P.qkv_rows + src + c.lane;
            unsigned long long raw[E];
#pragma unroll
            for (int e = 0; e < E; ++e) raw[e] = ll_get(qp + 32 * e);
            uint64_t t0 = 0;
            for (uint32_t i = 0;; ++i) {
                bool stale = false;
#pragma unroll
                for (int e = 0; e < E; ++e) stale |= (uint32_t)(raw[e] >> 32) != fqkv;
                if (!stale) break;
                t0 = poll_tick(c.P, &c.sh->abort, diag_of(c), i, t0, fqkv);
                if (t0 == ~0ull) return false;
#pragma unroll
                for (int e = 0; e < E; ++e)
                    if ((uint32_t)(raw[e] >> 32) != fqkv) raw[e] = ll_get(qp + 32 * e);
            }
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = __uint_as_float((uint32_t)raw[e]);
        }
        if (h <= GROUP) {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss += v[e] * v[e];
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)HD + P.eps);
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], inv), gn[e]);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                const float2 r = rp[e];
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
        if (!slot_wait_at(c, c.used, ks)) return false;
        if (!slot_wait_at(c, c.used + 1, vs)) return false;
#pragma unroll 1
        for (int half = 0; half < kKvChunk / (8 * kCWarps); ++half) {
        float sc[GROUP][8];
        float vv[8][D];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = (c.warp * (kKvChunk / (8 * kCWarps)) + half) * 8 + i;
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
        }
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
    // 3) merge the eight warps; a single split writes the output directly,
    //    otherwise it publishes its state and the last split merges them
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
    float* part = P.part + (((size_t)b * P.nkv + g) * (gridDim.x + 1) + split) * GROUP * (HD + 2);
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
        if (nsplit == 1) {
            const float o = A / L;
            const float o1 = __shfl_xor_sync(0xffffffffu, o, 1);
            if ((d & 1) == 0) put_pair(P.pl_o, P.nh * HD, b, (g * GROUP + h) * HD + d, o, o1, fatt);
        } else {
            part[h * (HD + 2) + d] = A;
            if (d == 0) {
                part[h * (HD + 2) + HD] = M;
                part[h * (HD + 2) + HD + 1] = L;
            }
        }
    }
    if (nsplit == 1) return cbar_sync(c);
    if (!cbar_sync(c)) return false;
    if (c.tid == 0) {
        __threadfence();  // the barrier made every thread's partial visible to this one
        const unsigned int old = atomicAdd(P.attn_cnt + ((size_t)l * P.bmax + b) * P.nkv + g, 1u);
        sh.flag_last = (old == (unsigned)(nsplit - 1));
        if (sh.flag_last) __threadfence();
    }
    if (!cbar_sync(c)) return false;
    if (sh.flag_last) {
        const float* p0 = P.part + (((size_t)b * P.nkv + g) * (gridDim.x + 1)) * GROUP * (HD + 2);
        for (int i = c.tid; i < GROUP * HD; i += kCThreads) {
            const int h = i / HD, d = i % HD;
            float M = -INFINITY;
            for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ld_cg_f32(p0 + ((size_t)s * GROUP + h) * (HD + 2) + HD));
            float L = 0.f, A = 0.f;
            for (int s = 0; s < nsplit; ++s) {
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
    int rot = (H / 16) % G;  // rotation of the QKV / gate-up / lm_head tiles

    // embedding gather (phase 0): x = E[tok] * s, planes of g_attn(0) * x
    {
        const int ntiles = H / 16;
        const uint32_t f = ep(0, kPhEmbed);
        for (int t = cta; t < ntiles; t += G) {
            for (int i = c.tid; i < B * 16; i += kCThreads) {
                const int b = i >> 4, r = i & 15, k = 16 * t + r;
                const int tok = P.tokens[b];
                const float v = (float)P.emb_raw[(size_t)tok * H + k] * P.emb_scale[tok];
                resid_store(c, t, r, b, v, false, P.gains[0]);
            }
            if (!finish_rows(c, t, P.pl_attn, P.ss_attn, f)) return;
            if (!cbar_sync(c)) return;
        }
        stamp(c, 1);
    }
    AttnSched as;
    as.init(B, P.nkv, G, sh.nchunk);
    if (c.tid < kMaxBatch) sh.best[c.tid] = 0ull;

    // Every phase of every layer, then the lm_head, runs through the same
    // loop body, so each piece of code exists once in the kernel: the
    // per-layer code walk then stays small enough for the instruction cache.
    const int nph = 5 * P.L + 1;
#pragma unroll 1
    for (int it = 0; it < nph; ++it) {
        const int l = it < 5 * P.L ? it / 5 : P.L - 1;
        const int ph = it < 5 * P.L ? kPhQkv + it % 5 : kPhLm;
        c.layer = it < 5 * P.L ? l : P.L;
        c.phase = ph;
        if (ph == kPhAtt) {
            for (int u = cta; u < as.U; u += G) {
                int b, g, split;
                as.locate(u, b, g, split);
                const int c0 = split * as.Q, c1 = min(sh.nchunk[b], c0 + as.Q);
                if (!attn_segment<HD, GROUP>(c, l, b, g, c0, c1, split, as.nsplit(b), ep(l, kPhQkv),
                                             ep(l, kPhAtt)))
                    return;
            }
            stamp(c, 2 + 6 * l + 1);
            continue;
        }
        // this phase's input and shape
        const bool rowtiles = ph == kPhO || ph == kPhDown;  // H-row tiles: split-K GEMV + residual
        const int K = ph == kPhO ? Dq : ph == kPhDown ? I : H;
        const int ntiles = rowtiles ? H / 16 : ph == kPhQkv ? P.qkv_rows / 16 : ph == kPhGu ? 2 * I / 16 : P.vpad / 16;
        const LLw* in = ph == kPhO ? P.pl_o : ph == kPhGu ? P.pl_ffn : ph == kPhDown ? P.pl_a : P.pl_attn;
        const uint32_t fin = (ph == kPhQkv || ph == kPhLm) ? (ph == kPhQkv && l == 0 ? ep(0, kPhEmbed)
                                                              : ep(ph == kPhQkv ? l - 1 : l, kPhDown))
                                                           : ep(l, ph - 1);
        const LLw* ss = ph == kPhO || ph == kPhDown ? nullptr : ph == kPhGu ? P.ss_ffn : P.ss_attn;
        const uint32_t fout = ph == kPhLm ? 0u : ep(l, ph);
        int t = rowtiles ? cta : first_tile(cta, rot, G);
        if (t < ntiles) {
            bool ok;
            if constexpr (NT == 1) ok = stage_plane(c, in, K, fin, ss, fin);
            else ok = ss ? load_rnorm(c, ss, fin) : true;
            if (!ok) return;
        }
        dstamp(c, 1);
        if (rowtiles) {
            const float* gain = ph == kPhO ? P.gains[4 * l + 1] : (l + 1 < P.L ? P.gains[4 * (l + 1)] : P.final_norm);
            LLw* plo = ph == kPhO ? P.pl_ffn : P.pl_attn;
            LLw* sso = ph == kPhO ? P.ss_ffn : P.ss_attn;
            constexpr int kEpi = (NT * 64 + kCThreads - 1) / kCThreads;  // epilogue items per thread
            for (; t < ntiles; t += G) {
                // this thread's gain values, fetched before the GEMV hides their latency
                float gv[kEpi];
#pragma unroll
                for (int j = 0; j < kEpi; ++j) {
                    const int i = c.tid + j * kCThreads;
                    const int rr = (((i & 63) >> 1) >> 2) + 8 * (i & 1);
                    gv[j] = i < NT * 64 ? gain[16 * t + rr] : 0.f;
                }
                if (!gemv_tile<NT>(c, K, in, fin)) return;
                dstamp(c, 2);
#pragma unroll
                for (int j = 0; j < kEpi; ++j) {
                    const int i = c.tid + j * kCThreads;
                    const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, b = 4 * n + (ln & 3);
                    if (i >= NT * 64 || b >= B) continue;
                    const int rr = (ln >> 2) + 8 * half;
                    const float v = sh.scl[rr] * red_sum<NT>(c, n, ln, half);
                    resid_store_g(c, t, rr, b, v, true, gv[j]);
                }
                if (!finish_rows(c, t, plo, sso, fout)) return;
                if (!cbar_sync(c)) return;
                dstamp(c, 3);
            }
        } else {
            const int mode = ph == kPhQkv ? kWmQkv : ph == kPhGu ? kWmGu : kWmLm;
            if constexpr (NT == 1) {
                if (!warp_tiles(c, mode, t, ntiles, G, H, fout)) return;
            } else {
                for (; t < ntiles; t += G) {
                    if (!gemv_tile<NT>(c, H, in, fin)) return;
                    dstamp(c, 2);
                    if (mode == kWmGu) {
                        for (int i = c.tid; i < NT * 32; i += kCThreads) {
                            const int n = i >> 5, ln = i & 31, gg = ln >> 2, b = 4 * n + (ln & 3);
                            if (b >= B) continue;
                            const float gate = sh.scl[gg] * sh.rnorm[b] * red_sum<NT>(c, n, ln, 0);
                            const float up = sh.scl[gg + 8] * sh.rnorm[b] * red_sum<NT>(c, n, ln, 1);
                            sh.gx[b][gg] = (gate / (1.0f + expf(-gate))) * up;
                        }
                        if (!cbar_sync(c)) return;
                        for (int i = c.tid; i < B * 4; i += kCThreads) {
                            const int b = i >> 2, jj = i & 3;
                            put_pair(P.pl_a, I, b, 8 * t + 2 * jj, sh.gx[b][2 * jj], sh.gx[b][2 * jj + 1], fout);
                        }
                    } else {
                        for (int i = c.tid; i < NT * 64; i += kCThreads) {
                            const int n = i >> 6, ln = (i & 63) >> 1, half = i & 1, b = 4 * n + (ln & 3);
                            if (b >= B) continue;
                            const int rr = (ln >> 2) + 8 * half, row = 16 * t + rr;
                            const float v = sh.scl[rr] * sh.rnorm[b] * red_sum<NT>(c, n, ln, half);
                            if (mode == kWmQkv) {
                                ll_put(P.qkv + (size_t)b * P.qkv_rows + row, __float_as_uint(v), fout);
                            } else if (row < P.vocab) {
                                if (P.logits) P.logits[(size_t)b * P.vocab + row] = v;
                                atomicMax(&sh.best[b], argmax_key(v, (uint32_t)row));
                            }
                        }
                    }
                    if (!cbar_sync(c)) return;
                    dstamp(c, 3);
                }
            }
            rot = (rot + ntiles) % G;
        }
        if (ph != kPhLm) stamp(c, 2 + 6 * l + (ph - kPhQkv));
    }
    // ---- argmax over the grid; the last CTA to finish closes the step
    if (!cbar_sync(c)) return;
    stamp(c, 2 + 6 * P.L);
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

// ------------------------------------------------------------------ layout of the dynamic shared memory
// [ring: ns slots][red: 8 x NT x 32 x 2 floats][stage (NT == 1): 2B x ld u32][full, empty mbarriers]
struct DynLayout {
    size_t ring, red, stage, bars, total;
    int stage_ld;
};

__host__ __device__ inline DynLayout dyn_layout(int ns, int NT, int B, int kmax) {
    DynLayout d;
    d.ring = 0;
    d.red = d.ring + (size_t)ns * kSlotBytes;
    d.stage = d.red + (size_t)kCWarps * NT * 64 * sizeof(float);
    d.stage_ld = kmax / 2 + kStagePad;
    const size_t stage_bytes = NT == 1 ? (size_t)2 * B * d.stage_ld * sizeof(uint32_t) : 0;
    d.bars = (d.stage + stage_bytes + 15) / 16 * 16;
    d.total = d.bars + 2 * (size_t)ns * sizeof(uint64_t);
    return d;
}

template <int NT, int HD, int GROUP>
__global__ void __launch_bounds__(kThreads, 1) persistent_step_kernel(PParams P) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ Shared sh;
    __shared__ PParams sP;
    if (threadIdx.x == 0) sP = P;
    const int ns = P.ns;
    const DynLayout dl = dyn_layout(ns, NT, P.B, P.kmax);
    Ctl c;
    c.P = &sP;
    c.sh = &sh;
    c.ring = dsm + dl.ring;
    c.red = reinterpret_cast<float*>(dsm + dl.red);
    c.stage = reinterpret_cast<uint32_t*>(dsm + dl.stage);
    c.stage_ld = dl.stage_ld;
    c.full = reinterpret_cast<uint64_t*>(dsm + dl.bars);
    c.empty = c.full + ns;
    c.ns = ns;
    c.used = 0;
    c.cphase = 0;
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    c.tid = threadIdx.x;
    c.layer = -1;
    c.phase = -1;
    c.dcount = 0;
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
    stamp(c, 0);
    consume<NT, HD, GROUP>(c);
    stamp(c, 3 + 6 * P.L);
    if (sh.abort && c.tid == 0) {
        // give every copy still in flight a bounded chance to land
        for (uint32_t i = 0; i < kSpinLimit && !sh.prod_done; ++i) __nanosleep(64);
        const uint32_t issued = sh.issued;
        for (uint32_t u = c.used; u < issued; ++u) mbar_wait_bounded(&c.full[u % ns], (u / ns) & 1);
    }
}

// ------------------------------------------------------------------ host side
static int nt_of(int B) { return B <= 4 ? 1 : B <= 8 ? 2 : B <= 16 ? 4 : 8; }

template <int NT, int HD, int GROUP>
static cudaError_t launch_t(const PParams& P, int grid, size_t smem, cudaStream_t st) {
    auto kern = persistent_step_kernel<NT, HD, GROUP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // shared-memory carveout just large enough (percent of the maximum), the rest stays L1
    const size_t need = smem + sizeof(Shared) + sizeof(PParams) + 1024;
    int carve = (int)((need * 100 + 232447) / 232448);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, carve > 100 ? 100 : carve);
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
    switch (nt_of(P.B)) {
        case 1: return launch_t<1, HD, GROUP>(P, grid, smem, st);
        case 2: return launch_t<2, HD, GROUP>(P, grid, smem, st);
        case 4: return launch_t<4, HD, GROUP>(P, grid, smem, st);
        default: return launch_t<8, HD, GROUP>(P, grid, smem, st);
    }
}

bool persistent_supported(const q3i8_dims& d) {
    const int group = d.n_heads / d.n_kv_heads;
    return (d.head_dim == 128 || d.head_dim == 64) && group == 2 && d.n_layers <= 127;
}

// Ring slots for batch B: as many as fit (at most kMaxSlots) after the
// static shared memory, the reduction buffer and the staged input.  The ring
// should hold more than one layer's share of a CTA's weight tiles (about ten
// 16.5 KB slots for the CTAs that also own O and down tiles), so that a
// layer's last weights are loaded before its consumers reach them.
int persistent_slots(int max_optin_smem, int B, int kmax) {
    const int nt = nt_of(B);
    const int fixed = (int)(sizeof(Shared) + sizeof(PParams)) + 1024;
    for (int ns = kMaxSlots; ns >= 2; --ns)
        if ((int)dyn_layout(ns, nt, B, kmax).total + fixed <= max_optin_smem) return ns;
    return 0;
}

cudaError_t launch_persistent_step(const PParams& P, int grid, cudaStream_t st) {
    const size_t smem = dyn_layout(P.ns, nt_of(P.B), P.B, P.kmax).total;
    if (P.hd == 128) return launch_hg<128, 2>(P, grid, smem, st);
    return launch_hg<64, 2>(P, grid, smem, st);
}

}  // namespace q3
