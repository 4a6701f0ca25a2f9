// q3i8_op_attention_static: split-KV decode attention whose partial softmax
// states go to a scratch array compiled into the library, so that a call
// allocates no device memory.  Meant for callers that have no device
// allocator to hand (a plain C host program) or must not call
// cudaMalloc/cudaFree between steps (cudaFree synchronises the device).
#include <mutex>
#include <stdio.h>

#include "../../include/q3i8.h"
#include "kernels.h"

int q3_report_error(int code, const char* msg);  // engine.cu

using q3::attn_part_bytes;
using q3::launch_attention;

namespace {

constexpr size_t kScratchBytes = Q3I8_OP_ATTENTION_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices];    // device address of the scratch, per device
void* g_scratch_ctx[kMaxDevices];     // the context that address belongs to

// The current driver context (reached through the runtime's driver entry
// point, so the library needs no link against the driver library).  A device
// reset or a released primary context gives the device a new context whose
// module copy of the scratch lives elsewhere, so the address is looked up
// again whenever the context changes.
void* current_context() {
    typedef int (*GetCurrentFn)(void**);
    static GetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<GetCurrentFn>(p);
    });
    void* ctx = nullptr;
    if (fn && fn(&ctx) != 0) ctx = nullptr;
    return ctx;
}

int report(int code, const char* fmt, long long a = 0, long long b = 0) {
    char buf[256];
    snprintf(buf, sizeof buf, fmt, a, b);
    return q3_report_error(code, buf);
}

}  // namespace

// The scratch itself: one copy per device, in the module's static memory.
// Each (row, head, split) state is written by the split kernel before the
// merge kernel reads it, so its contents never need clearing.
static __device__ __align__(256) float g_attn_scratch[kScratchBytes / sizeof(float)];

// Device address of g_attn_scratch on the current device, looked up with
// that device current the first time and again whenever its context changed.
static int scratch_on_current_device(float** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report(Q3_ERR_NO_DEVICE, "op_attention_static: no current device");
    if (dev < 0 || dev >= kMaxDevices)
        return report(Q3_ERR_INVALID_ARGUMENTS, "op_attention_static: device %lld beyond the %lld supported", dev,
                      kMaxDevices);
    void* ctx = current_context();  // null before the runtime made one current: then looked up below
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev] || ctx != g_scratch_ctx[dev]) {
        g_scratch_ptr[dev] = nullptr;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || !p) {
            char buf[256];
            snprintf(buf, sizeof buf, "op_attention_static: scratch lookup failed: %s", cudaGetErrorString(e));
            return q3_report_error(Q3_ERR_CUDA, buf);
        }
        g_scratch_ptr[dev] = (float*)p;
        g_scratch_ctx[dev] = current_context();  // the lookup made the device's context current
    }
    *out = g_scratch_ptr[dev];
    return Q3_OK;
}

extern "C" int q3i8_op_attention_static(const float* q, const uint16_t* k, const uint16_t* v, const int32_t* row_seq,
                                        const int32_t* row_len, int32_t R, int32_t n_heads, int32_t n_kv_heads,
                                        int32_t hd, int32_t cap, int32_t splits, float* out, int32_t* d_status,
                                        void* cuda_stream) {
    if (!q || !k || !v || !row_seq || !row_len || !out)
        return report(Q3_ERR_INVALID_ARGUMENTS, "op_attention_static: NULL pointer");
    if (R < 1 || n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || (hd != 64 && hd != 128) || cap < 64 ||
        cap % 64 || splits < 1 || splits > 64)
        return report(Q3_ERR_INVALID_ARGUMENTS, "op_attention_static: unsupported sizes");
    if (((uintptr_t)k & 15) || ((uintptr_t)v & 15))
        return report(Q3_ERR_INVALID_ARGUMENTS, "op_attention_static: K/V caches must be 16-byte aligned");
    const size_t need = attn_part_bytes(R, n_heads, hd, splits);
    if (need > kScratchBytes)
        return report(Q3_ERR_INVALID_ARGUMENTS,
                      "op_attention_static: these sizes need %lld bytes of scratch, above the static limit of %lld "
                      "bytes (use q3i8_op_attention with a workspace)",
                      (long long)need, (long long)kScratchBytes);
    float* scratch = nullptr;
    int rc = scratch_on_current_device(&scratch);
    if (rc) return rc;
    rc = launch_attention(q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, row_seq, row_len, 0, R, n_heads,
                          n_kv_heads, hd, cap, splits, scratch, out, nullptr, 0, d_status, (cudaStream_t)cuda_stream);
    if (rc) return report(Q3_ERR_INVALID_ARGUMENTS, "op_attention_static: unsupported head_dim/group");
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char buf[256];
        snprintf(buf, sizeof buf, "op_attention_static launch: %s", cudaGetErrorString(e));
        return q3_report_error(Q3_ERR_CUDA, buf);
    }
    return Q3_OK;
}
