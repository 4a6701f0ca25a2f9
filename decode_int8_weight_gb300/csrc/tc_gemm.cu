// Prefill projections on the 5th-generation tensor cores (tcgen05 + TMEM).
//
//   Y[m][n] = s[n] * sum_k q[n][k] * x[m][k]     (m: prompt rows, n: outputs)
//
// The activations arrive as f16 hi/lo planes (x = hi + lo, about 22
// significant bits), stored so that row m of the [M][2K] view is hi(m, :)
// followed by lo(m, :).  Every k-tile of 64 therefore runs two MMAs against
// one weight tile: hi x W and lo x W, accumulating in fp32 in TMEM.  int8
// weights are exact in f16.
//
// One CTA computes a 128 x 128 output tile:
//   warp 0     TMA producer: per stage, the hi and lo activation tiles
//              (128 x 64 f16, 128-byte swizzle) and the int8 weight tile
//              (128 x 64 bytes) into a 4-stage ring;
//   warp 1     allocates 128 TMEM columns; one thread issues the MMAs
//              (M = 128, N = 128, K = 16 each) and commits each stage back
//              to the producer;
//   warps 2-5  convert the int8 weight tile to f16 in the 128-byte swizzled
//              K-major layout the MMA descriptor reads, then run the
//              epilogue from TMEM (tcgen05.ld): scale, and store / add to
//              the residual / SiLU-gate into hi/lo planes.
// Every wait is bounded; a wait that gives up sets the status word and the
// CTA winds down (copies drained, TMEM freed).
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)
#include <stdio.h>

#include "common.cuh"
#include "kernels.h"

namespace q3 {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kStages = 4;
constexpr int kTcThreads = 192;
constexpr uint32_t kATile = kBM * kBK * 2;     // 16 KB f16, one of hi / lo
constexpr uint32_t kB16Tile = kBN * kBK * 2;   // 16 KB f16 weights (converted)
constexpr uint32_t kB8Tile = kBN * kBK;        // 8 KB int8 weights (as loaded)
constexpr uint32_t kStageBytes = 2 * kATile + kB16Tile + kB8Tile;  // 56 KB, a multiple of 1024
constexpr uint32_t kTxBytes = 2 * kATile + kB8Tile;                // bytes the TMA lands per stage
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + 256;

struct TcArgs {
    const float* scale;
    int M, N, K, mode;
    float* y;
    int ldy;
    __half* yh;
    int ldyh;
    int32_t* status;
    int splits;    // K split over gridDim.z CTAs (1: the CTA finishes its tile itself)
    float* part;   // splits > 1: [splits][M][N] fp32 partial sums, unscaled
};

// The output epilogue of 16 consecutive columns n .. n + 15 of row m, from
// their scaled fp32 values: store, add to the residual, or (a 16-row group
// of the fused gate/up matrix: 8 gate rows, then the 8 up rows of the same
// units) SiLU-gate into hi/lo planes.
Q3_DEV void epilogue16(const TcArgs& g, int m, int n, const float (&v)[16]) {
    if (g.mode == kSiluGate) {
        const int u0 = n >> 1;
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const float a0 = (v[i] / (1.0f + expf(-v[i]))) * v[8 + i];
            const float a1 = (v[i + 1] / (1.0f + expf(-v[i + 1]))) * v[9 + i];
            __half h0, l0, h1, l1;
            split_f16(a0, h0, l0);
            split_f16(a1, h1, l1);
            hw[i / 2] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            lw[i / 2] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
        }
        *reinterpret_cast<uint4*>(g.yh + (size_t)(2 * m) * g.ldyh + u0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(g.yh + (size_t)(2 * m + 1) * g.ldyh + u0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    } else {
        float4* dst = reinterpret_cast<float4*>(g.y + (size_t)m * g.ldy + n);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 o = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            if (g.mode == kResid) {
                const float4 p = dst[i];
                o.x += p.x, o.y += p.y, o.z += p.z, o.w += p.w;
            }
            dst[i] = o;
        }
    }
}

// ------------------------------------------------------------------ PTX wrappers
Q3_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

Q3_DEV void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
Q3_DEV void tc_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
Q3_DEV void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
Q3_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
Q3_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (TMEM) [+]= A (smem) x B (smem)^T, f16 inputs, fp32 accumulate.
Q3_DEV void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on bar when every MMA this thread issued so far has completed.
Q3_DEV void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
Q3_DEV void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
Q3_DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

Q3_DEV void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// Shared-memory matrix descriptor: K-major tile, 128-byte rows, 128-byte
// swizzle, 8-row groups 1024 bytes apart (tile base 1024-byte aligned).
Q3_DEV uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4)  // start address / 16
           | (1ull << 16)                      // leading offset (unused by swizzled K-major)
           | (64ull << 32)                     // stride offset: 1024 bytes / 16
           | (1ull << 46)                      // descriptor version of this architecture
           | (2ull << 61);                     // layout: 128-byte swizzle
}

// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, both
// K-major, N = kBN, M = kBM.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

Q3_DEV bool wait_or_flag(uint64_t* bar, uint32_t parity, int32_t* status, volatile int* abort_sm) {
    if (*abort_sm) return false;
    if (mbar_wait_bounded(bar, parity)) return true;
    *abort_sm = 1;
    set_status(status, kStatusTimeout);
    return false;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcArgs g) {
    extern __shared__ uint8_t dsm[];
    const uint32_t raw = smem_u32(dsm);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = dsm + (base - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(gbase + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* bready = empty + kStages;
    uint64_t* done = bready + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_sm = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
    // this CTA's k-tiles [kt0, kt0 + NK) of the K / kBK
    const int KT = g.K / kBK, kt0 = (int)blockIdx.z * KT / g.splits;
    const int NK = ((int)blockIdx.z + 1) * KT / g.splits - kt0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&bready[s], 4);
        }
        mbar_init(done, 1);
        *abort_sm = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc_alloc(smem_u32(tmem_slot), kBN);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < NK; ++kt) {
                const int s = kt % kStages;
                if (kt >= kStages && !wait_or_flag(&empty[s], ((kt / kStages) - 1) & 1, g.status, abort_sm)) break;
                const uint32_t st = base + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kTxBytes);
                const int kx = (kt0 + kt) * kBK;
                tma_load_2d(st, &tmA, kx, m0, smem_u32(&full[s]));                 // hi
                tma_load_2d(st + kATile, &tmA, g.K + kx, m0, smem_u32(&full[s]));  // lo
                tma_load_2d(st + 2 * kATile + kB16Tile, &tmB, kx, n0, smem_u32(&full[s]));
                issued = kt + 1;
            }
            // every copy this thread started has landed before the CTA can end
            for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt)
                mbar_wait_bounded(&full[kt % kStages], (kt / kStages) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int kt = 0; kt < NK; ++kt) {
                const int s = kt % kStages;
                if (!wait_or_flag(&bready[s], (kt / kStages) & 1, g.status, abort_sm)) break;
                tc_fence_after();
                const uint32_t st = base + s * kStageBytes;
                const uint64_t dh = sw128_desc(st), dl = sw128_desc(st + kATile), db = sw128_desc(st + 2 * kATile);
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j) {
                    // a 16-wide k step is 32 bytes along the swizzled row: +2 in the address field
                    tc_mma(tmem, dh + 2 * j, db + 2 * j, kIdesc, (kt | j) != 0);
                    tc_mma(tmem, dl + 2 * j, db + 2 * j, kIdesc, 1u);
                }
                tc_commit(smem_u32(&empty[s]));
            }
            tc_commit(smem_u32(done));
            mbar_wait_bounded(done, 0);  // the MMAs are finished before TMEM can be freed
        }
    } else {
        const int ct = threadIdx.x - 64;  // 0 .. 127
        for (int kt = 0; kt < NK; ++kt) {
            const int s = kt % kStages;
            if (!wait_or_flag(&full[s], (kt / kStages) & 1, g.status, abort_sm)) break;
            const uint32_t st = base + s * kStageBytes;
            const uint32_t b16 = st + 2 * kATile, b8 = b16 + kB16Tile;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                // 16 weights of one row: row = j / 4, bytes 16 * (j % 4) .. + 15
                const int j = ct + 128 * r, row = j >> 2, q = j & 3;
                const uint4 w = lds128(b8 + row * 64 + q * 16);
                uint32_t f[8];
                u8x4_to_f16x2x2(w.x ^ 0x80808080u, f[0], f[1]);  // signed -> biased bytes, then exact f16
                u8x4_to_f16x2x2(w.y ^ 0x80808080u, f[2], f[3]);
                u8x4_to_f16x2x2(w.z ^ 0x80808080u, f[4], f[5]);
                u8x4_to_f16x2x2(w.w ^ 0x80808080u, f[6], f[7]);
                const uint32_t rb = b16 + row * 128;
                sts128(rb + ((((uint32_t)(2 * q)) ^ (row & 7)) << 4), f[0], f[1], f[2], f[3]);
                sts128(rb + ((((uint32_t)(2 * q + 1)) ^ (row & 7)) << 4), f[4], f[5], f[6], f[7]);
            }
            fence_proxy_async_smem();  // the MMA reads these through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&bready[s]);
        }
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. rows of this tile
        if (wait_or_flag(done, 0, g.status, abort_sm)) {
            tc_fence_after();
            const int qd = warp & 3;
            const int m = m0 + 32 * qd + lane;
#pragma unroll 1
            for (int c = 0; c < kBN; c += 16) {
                uint32_t r[16];
                tc_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)c, r);
                tc_wait_ld();
                if (m >= g.M) continue;
                const int n = n0 + c;
                float v[16];
                if (g.splits > 1) {
                    // unscaled partial sums; the reduction scales and finishes them
                    float4* dst = reinterpret_cast<float4*>(g.part + ((size_t)blockIdx.z * g.M + m) * g.N + n);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                             __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                    continue;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]) * __ldg(g.scale + n + i);
                epilogue16(g, m, n, v);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kBN);
    }
}

// Split-K: thread (m, 16-column group) sums the splits' partials in split
// order (the result does not depend on which CTA finished first), scales
// and runs the epilogue.
__global__ void __launch_bounds__(256) tc_splitk_reduce(TcArgs g) {
    const int groups = g.N / 16;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)g.M * groups) return;
    const int m = (int)(i / groups), n = (int)(i - (long long)m * groups) * 16;
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = 0.f;
    for (int z = 0; z < g.splits; ++z) {
        const float4* src = reinterpret_cast<const float4*>(g.part + ((size_t)z * g.M + m) * g.N + n);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 p = __ldcg(src + q);
            v[4 * q] += p.x, v[4 * q + 1] += p.y, v[4 * q + 2] += p.z, v[4 * q + 3] += p.w;
        }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] *= __ldg(g.scale + n + j);
    epilogue16(g, m, n, v);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

bool tc_gemm_supported(int N, int K) { return N > 0 && K > 0 && N % kBN == 0 && K % kBK == 0; }

// K splits of an M x N x K projection when the output tiles alone leave
// more than half of the SMs idle: as many as fit in one wave (a second,
// partial wave would leave most SMs idle at its end), each split keeping
// at least 4 k-tiles.
int tc_gemm_splits(int M, int N, int K, int num_sms) {
    const int tiles = (M + kBM - 1) / kBM * (N / kBN);
    if (tiles * 2 > num_sms) return 1;
    int s = num_sms / tiles;
    s = s < 8 ? s : 8;
    const int cap = (K / kBK) / 4;
    s = s < cap ? s : cap;
    return s > 1 ? s : 1;
}

size_t tc_gemm_work_bytes(int M, int N, int K, int num_sms) {
    const int s = tc_gemm_splits(M, N, K, num_sms);
    return s > 1 ? (size_t)s * M * N * 4 : 0;
}

int launch_tc_gemm(const __half* a_planes, const int8_t* w, const float* scale, int M, int N, int K, int mode,
                   float* y, int ldy, __half* yh, int ldyh, int32_t* status, cudaStream_t st, float* work,
                   size_t work_bytes, int num_sms) {
    if (M <= 0) return 0;
    if (!tc_gemm_supported(N, K) || (mode != kStore && mode != kResid && mode != kSiluGate)) return -1;
    if (((uintptr_t)a_planes & 15) || ((uintptr_t)w & 15) || (mode == kSiluGate ? (ldyh % 8 != 0) : (ldy % 4 != 0)))
        return -1;
    EncodeTiledFn enc = encoder();
    if (!enc) return -2;
    CUtensorMap ta, tb;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(2 * K), (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)(2 * K) * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a_planes), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return -3;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBN};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(w), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return -3;
    }
    if (allow_max_dynamic_smem((const void*)tc_gemm_kernel) != cudaSuccess) return -4;
    int splits = num_sms > 0 ? tc_gemm_splits(M, N, K, num_sms) : 1;
    if (splits > 1 && (!work || work_bytes < (size_t)splits * M * N * 4 || ((uintptr_t)work & 15))) splits = 1;
    TcArgs g{scale, M, N, K, mode, y, ldy, yh, ldyh, status, splits, work};
    const dim3 grid(N / kBN, (M + kBM - 1) / kBM, splits);
    tc_gemm_kernel<<<grid, kTcThreads, kSmemBytes, st>>>(ta, tb, g);
    if (splits > 1) {
        const long long n = (long long)M * (N / 16);
        tc_splitk_reduce<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(g);
    }
    return 0;
}

}  // namespace q3
