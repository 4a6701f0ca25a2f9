// Causal prefill attention on tensor cores (flash-attention form).
//
// One CTA takes 32 consecutive prompt positions of one sequence and one kv
// head, i.e. both query heads of the group (GROUP == 2) x 32 rows; each of
// its 4 warps owns 16 rows of one head.  K/V tiles of 64 positions are
// staged in shared memory (cp.async, double buffered, rows padded to 272
// bytes so that fragment loads are free of bank conflicts) and every tile
// serves both heads.
//
// Scores S = Q K^T and the output P V run on bf16 mma.sync with fp32
// accumulation.  K and V are bf16 in the cache, hence exact operands; the
// fp32 queries and probabilities are split into bf16 hi + lo parts (about 16
// significant bits together) and multiplied twice, so the result stays
// within fp32 rounding of the plain definition: softmax over positions
// 0..p (the current one included) of q.k / sqrt(hd), times V.  The softmax
// runs online over the tiles (running max and sum per row, fp32, expf).
//
// Output: hi/lo f16 planes of o, planes[(2r + part) * ldh + head * hd + d]
// for flat prompt row r -- the operand layout of the O projection.
#include "common.cuh"
#include "kernels.h"

namespace q3 {
namespace {

constexpr int kQRows = 32;   // prompt positions per CTA
constexpr int kKT = 64;      // positions per K/V tile
constexpr int kHD = 128;     // head dim of this kernel
constexpr int kRowB = kHD * 2 + 16;  // padded smem row: 272 bytes
constexpr int kTileB = kKT * kRowB;  // 17408 bytes per K or V tile
constexpr int kPfThreads = 128;
constexpr size_t kPfSmem = 2 * 2 * (size_t)kTileB;  // 2 stages x (K, V)

Q3_DEV void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
Q3_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
Q3_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

Q3_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
Q3_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

Q3_DEV void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// {x, y} -> bf16x2 hi part and the bf16x2 of the remainders
Q3_DEV void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat16 hx = __float2bfloat16_rn(x), hy = __float2bfloat16_rn(y);
    const __nv_bfloat16 lx = __float2bfloat16_rn(x - __bfloat162float(hx));
    const __nv_bfloat16 ly = __float2bfloat16_rn(y - __bfloat162float(hy));
    hi = (uint32_t)__bfloat16_as_ushort(hx) | ((uint32_t)__bfloat16_as_ushort(hy) << 16);
    lo = (uint32_t)__bfloat16_as_ushort(lx) | ((uint32_t)__bfloat16_as_ushort(ly) << 16);
}

Q3_DEV uint32_t pack_h2(float a, float b) {
    return (uint32_t)__half_as_ushort(__float2half_rn(a)) | ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
}

// blocks[i] = {sequence, first position, flat row of position 0, length}
__global__ void __launch_bounds__(kPfThreads, 2)
    attn_prefill_kernel(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, const int4* blocks, int nh,
                        int nkv, int cap, __half* outh, int ldh) {
    extern __shared__ __align__(16) uint8_t sm[];
    const int4 blk = blocks[blockIdx.x];
    const int b = blk.x, p0 = blk.y, row0 = blk.z, len = blk.w;
    const int g = blockIdx.y;  // kv head
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gg = lane >> 2, t = lane & 3;
    const int head = 2 * g + (warp >> 1);
    const int pw = p0 + 16 * (warp & 1);  // first position of this warp's rows
    const size_t kvbase = (((size_t)b * nkv + g) * cap) * kHD;
    const float scale = 1.0f / sqrtf((float)kHD);

    // queries of rows pw + gg and pw + gg + 8 (positions past the prompt read row pw)
    uint32_t qh[8][4], ql[8][4];
    {
        const int pa = pw + gg < len ? pw + gg : pw, pb = pw + gg + 8 < len ? pw + gg + 8 : pw;
        const float* qa = q + ((size_t)(row0 + pa) * nh + head) * kHD;
        const float* qb = q + ((size_t)(row0 + pb) * nh + head) * kHD;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const float2 x0 = *reinterpret_cast<const float2*>(qa + 16 * kk + 2 * t);
            const float2 x1 = *reinterpret_cast<const float2*>(qb + 16 * kk + 2 * t);
            const float2 x2 = *reinterpret_cast<const float2*>(qa + 16 * kk + 2 * t + 8);
            const float2 x3 = *reinterpret_cast<const float2*>(qb + 16 * kk + 2 * t + 8);
            split_bf16x2(x0.x * scale, x0.y * scale, qh[kk][0], ql[kk][0]);
            split_bf16x2(x1.x * scale, x1.y * scale, qh[kk][1], ql[kk][1]);
            split_bf16x2(x2.x * scale, x2.y * scale, qh[kk][2], ql[kk][2]);
            split_bf16x2(x3.x * scale, x3.y * scale, qh[kk][3], ql[kk][3]);
        }
    }

    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    const uint32_t sbase = smem_u32(sm);
    const int last_pos = min(p0 + kQRows, len) - 1;  // last query position of the CTA
    const int ntiles = last_pos / kKT + 1;

    // stage tile i (positions 64 i ..) into buffer i & 1; rows past the prompt are zero
    auto stage = [&](int i) {
        const uint32_t kb = sbase + (uint32_t)((i & 1) * 2 * kTileB), vb = kb + kTileB;
        for (int c = threadIdx.x; c < kKT * 16; c += kPfThreads) {
            const int r = c >> 4, ch = c & 15;
            const int pos = i * kKT + r;
            const uint32_t off = (uint32_t)(r * kRowB + ch * 16);
            if (pos < len) {
                cp_async16(kb + off, kc + kvbase + (size_t)pos * kHD + ch * 8);
                cp_async16(vb + off, vc + kvbase + (size_t)pos * kHD + ch * 8);
            } else {
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(kb + off), "r"(0u) : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vb + off), "r"(0u) : "memory");
            }
        }
        cp_async_commit();
    };

    stage(0);
    for (int i = 0; i < ntiles; ++i) {
        if (i + 1 < ntiles) {
            stage(i + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int k0 = i * kKT;
        if (k0 <= pw + 15) {  // this warp's rows see some key of the tile
            const uint32_t kb = sbase + (uint32_t)((i & 1) * 2 * kTileB), vb = kb + kTileB;
            // S = Q K^T for 16 rows x 64 keys
            float s[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    // matrices: keys 8j.. / dims 16kk, +8 ; keys 8(j+1).. / dims 16kk, +8
                    const int mi = lane >> 3, r = lane & 7;
                    const int key = 8 * (j + (mi >> 1)) + r, dim = 16 * kk + 8 * (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + (uint32_t)(key * kRowB + dim * 2), b0, b1, b2, b3);
                    mma_bf16(s[j], qh[kk], b0, b1);
                    mma_bf16(s[j], ql[kk], b0, b1);
                    mma_bf16(s[j + 1], qh[kk], b2, b3);
                    mma_bf16(s[j + 1], ql[kk], b2, b3);
                }
            }
            // causal mask and online softmax; rows pw + gg (e = 0, 1) and pw + gg + 8 (e = 2, 3)
            float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = k0 + 8 * j + 2 * t + (e & 1);
                    const int qp = pw + gg + 8 * (e >> 1);
                    if (key > qp) s[j][e] = -INFINITY;
                    mx[e >> 1] = fmaxf(mx[e >> 1], s[j][e]);
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            }
            float corr[2], rs[2] = {0.f, 0.f};
#pragma unroll
            for (int h = 0; h < 2; ++h) corr[h] = mrow[h] == -INFINITY ? 0.f : expf(mrow[h] - mx[h]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pe = s[j][e] == -INFINITY ? 0.f : expf(s[j][e] - mx[e >> 1]);
                    s[j][e] = pe;
                    rs[e >> 1] += pe;
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 1);
                rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 2);
                lrow[h] = lrow[h] * corr[h] + rs[h];
                mrow[h] = mx[h];
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                o[j][0] *= corr[0], o[j][1] *= corr[0];
                o[j][2] *= corr[1], o[j][3] *= corr[1];
            }
            // O += P V: k-step kk covers keys 16kk .. 16kk + 15 (score tiles 2kk, 2kk + 1)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t ph[4], pl[4];
                split_bf16x2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
                split_bf16x2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
                split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
                split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    // matrices: keys 16kk.., +8 / dims 8j ; keys 16kk.., +8 / dims 8(j+1)
                    const int mi = lane >> 3, r = lane & 7;
                    const int key = 16 * kk + 8 * (mi & 1) + r, dim = 8 * (j + (mi >> 1));
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + (uint32_t)(key * kRowB + dim * 2), b0, b1, b2, b3);
                    mma_bf16(o[j], ph, b0, b1);
                    mma_bf16(o[j], pl, b0, b1);
                    mma_bf16(o[j + 1], ph, b2, b3);
                    mma_bf16(o[j + 1], pl, b2, b3);
                }
            }
        }
        __syncthreads();  // the buffer is refilled two tiles later
    }

    // o / l -> hi/lo f16 planes
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int p = pw + gg + 8 * h;
        if (p >= len) continue;
        const float inv = 1.0f / lrow[h];
        const size_t r = (size_t)row0 + p;
        __half* dh = outh + (2 * r) * ldh + head * kHD;
        __half* dl = outh + (2 * r + 1) * ldh + head * kHD;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float v0 = o[j][2 * h] * inv, v1 = o[j][2 * h + 1] * inv;
            __half h0, l0, h1, l1;
            split_f16(v0, h0, l0);
            split_f16(v1, h1, l1);
            const int d = 8 * j + 2 * t;
            *reinterpret_cast<uint32_t*>(dh + d) =
                (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            *reinterpret_cast<uint32_t*>(dl + d) =
                (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
        }
    }
}

}  // namespace

bool attn_prefill_supported(int nh, int nkv, int hd) { return hd == kHD && nkv > 0 && nh == 2 * nkv; }

int attn_prefill_blocks(const int32_t* lens, int B, int4* out, int cap_blocks, const int32_t* slots) {
    int n = 0, row0 = 0;
    for (int b = 0; b < B; ++b) {
        for (int p = 0; p < lens[b]; p += kQRows) {
            if (n < cap_blocks) out[n] = make_int4(slots ? slots[b] : b, p, row0, lens[b]);
            ++n;
        }
        row0 += lens[b];
    }
    return n;
}

int launch_attn_prefill(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, const int4* blocks,
                        int nblocks, int nh, int nkv, int hd, int cap, __half* outh, int ldh, cudaStream_t st) {
    if (nblocks <= 0) return 0;
    if (!attn_prefill_supported(nh, nkv, hd) || cap % kKT) return -1;
    if (allow_max_dynamic_smem((const void*)attn_prefill_kernel) != cudaSuccess) return -2;
    attn_prefill_kernel<<<dim3(nblocks, nkv), kPfThreads, kPfSmem, st>>>(q, kc, vc, blocks, nh, nkv, cap, outh, ldh);
    return 0;
}

}  // namespace q3
