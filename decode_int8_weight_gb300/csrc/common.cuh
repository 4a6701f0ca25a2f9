// Device helpers shared by the q3i8 kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define Q3_DEV __device__ __forceinline__

namespace q3 {

// Limits of every bounded device wait: a poll count (iterations of a
// try_wait/poll loop with a short sleep) and a wall time, whichever runs out
// first.  Both sit far above any legitimate wait (microseconds).  After one
// runs out a kernel records Q3 status 7 and returns.
constexpr uint32_t kSpinLimit = 1u << 22;
constexpr uint64_t kWaitWallNs = 1000000000ull;
constexpr int kStatusTimeout = 7;

// ------------------------------------------------------------- conversions

// One 32-bit word of four biased weights (u = q + 128) -> two f16x2 words:
// lo = {q0, q1}, hi = {q2, q3}, exact.  0x64 in the high byte of an f16
// makes 1024 + u; subtracting 1152 leaves q.
Q3_DEV void u8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t magic = 0x64806480u;  // f16 1152 in both halves
    uint32_t a = __byte_perm(w, 0x64646464u, 0x4140);
    uint32_t b = __byte_perm(w, 0x64646464u, 0x4342);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(magic));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(magic));
}

// Same bytes -> f16x2 words {1024 + u0, 1024 + u1}, {1024 + u2, 1024 + u3}:
// one byte permute per pair and no subtraction.  A GEMV fed these operands
// computes sum (q + 1152) x = (W . x) + 1152 * sum x; the caller subtracts
// 1152 * sum x once per output.
Q3_DEV void u8x4_to_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
    lo = __byte_perm(w, 0x64646464u, 0x4140);
    hi = __byte_perm(w, 0x64646464u, 0x4342);
}
constexpr float kBias = 1152.0f;

// v = hi + lo with hi = f16(v), lo = f16(v - hi): about 22 significant bits.
Q3_DEV void split_f16(float v, __half& hi, __half& lo) {
    hi = __float2half_rn(v);
    lo = __float2half_rn(v - __half2float(hi));
}

Q3_DEV float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Order-preserving map of a float to uint32 (larger float -> larger key).
Q3_DEV uint32_t float_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// 64-bit argmax key: maximum value first, then the LOWEST index.
Q3_DEV unsigned long long argmax_key(float v, uint32_t idx) {
    return ((unsigned long long)float_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

Q3_DEV uint32_t argmax_key_index(unsigned long long k) { return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull); }

// ------------------------------------------------------------- tensor core
// mma.sync m16n8k16, f16 inputs, fp32 accumulate (A row-major, B col-major).
Q3_DEV void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------- loads
Q3_DEV uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ------------------------------------------------------------- mbarrier + bulk copy
Q3_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

Q3_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

Q3_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

Q3_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

Q3_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

Q3_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

Q3_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

Q3_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase: at most `limit` polls and about
// kWaitWallNs of wall time (read every 256 polls); false if either ran out
// (limit 0 gives up at once).
Q3_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit = kSpinLimit) {
    uint64_t t0 = 0;
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitWallNs) return false;
        }
        if (i > 64) __nanosleep(64);
    }
    return false;
}

// 1-D bulk copy global -> shared, completion counted on bar (bytes % 16 == 0,
// both addresses 16-byte aligned).
Q3_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Ask L2 to fetch [p, p + bytes) from global memory; nothing is returned to
// the SM (p 16-byte aligned, bytes a multiple of 16).
Q3_DEV void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------- shared-memory loads
// Explicit shared-space loads (32-bit shared addresses), so that hot loops
// never go through generic addressing.
Q3_DEV uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
Q3_DEV uint32_t lds32(uint32_t a) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
    return r;
}
Q3_DEV float lds_f32(uint32_t a) {
    float r;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(a));
    return r;
}
Q3_DEV uint2 lds64(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}

// ------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while
// the previous kernel in the stream is still running.  It lets its own
// successor be scheduled at once (pdl_launch_dependents) and waits until
// every kernel it depends on has completed and its writes are visible
// (pdl_wait) before touching memory.  Both are no-ops for a plain launch.
Q3_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
Q3_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------- clusters
Q3_DEV int cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return (int)r;
}
Q3_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
Q3_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// The same object in the shared memory of CTA `rank` of this cluster.
template <typename T>
Q3_DEV const T* peer(const T* p, int rank) {
    return cooperative_groups::this_cluster().map_shared_rank(p, rank);
}

// ------------------------------------------------------------- misc
Q3_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

Q3_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

Q3_DEV void set_status(int32_t* st, int code) {
    if (st) atomicCAS(st, 0, code);
}

}  // namespace q3
