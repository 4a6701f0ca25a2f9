// q3i8_op_wait_probe: runs the bounded mbarrier wait that every kernel of the
// library uses (mbar_wait_bounded) on a barrier phase that completes only
// when the caller asks for it, with a caller-chosen poll limit.  With the
// phase left open the wait must run out, set the device status to the
// time-out code and return, leaving the context usable; this is how the
// give-up path of the waits is exercised without faulting or hanging a GPU.
#include <stdio.h>

#include "../../include/q3i8.h"
#include "common.cuh"

int q3_report_error(int code, const char* msg);  // engine.cu

namespace {

using namespace q3;

static_assert(kStatusTimeout == Q3_ERR_TIMEOUT, "device time-out code and the ABI's differ");

// One CTA of one warp.  The barrier expects one arrival; thread 0 makes it
// only when `arrive` is set, so otherwise phase 0 never completes.  Every
// thread waits on phase 0; each one that gives up marks the status.  No
// asynchronous copy targets the barrier, so returning with it still open
// leaves nothing in flight.
__global__ void wait_probe_kernel(int arrive, uint32_t limit, int32_t* status, unsigned long long* elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait_bounded(&bar, 0, limit);
    const uint64_t t1 = globaltimer_ns();
    if (!ok) set_status(status, kStatusTimeout);
    if (threadIdx.x == 0 && elapsed_ns) *elapsed_ns = t1 - t0;
}

int cuda_fail(const char* what, cudaError_t e) {
    char buf[256];
    snprintf(buf, sizeof buf, "op_wait_probe %s: %s", what, cudaGetErrorString(e));
    return q3_report_error(Q3_ERR_CUDA, buf);
}

}  // namespace

extern "C" int q3i8_op_wait_probe(int32_t arrive, int32_t limit, int32_t* d_status, uint64_t* d_elapsed_ns,
                                  void* cuda_stream) {
    if (!d_status) return q3_report_error(Q3_ERR_INVALID_ARGUMENTS, "op_wait_probe: d_status is NULL");
    const uint32_t polls = limit < 0 ? q3::kSpinLimit : (uint32_t)limit;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    cudaError_t e = cudaMemsetAsync(d_status, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_fail("status reset", e);
    wait_probe_kernel<<<1, 32, 0, st>>>(arrive != 0, polls, d_status, (unsigned long long*)d_elapsed_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail("launch", e);
    int32_t h = 0;
    e = cudaMemcpyAsync(&h, d_status, sizeof h, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail("status read", e);
    if (h == Q3_ERR_TIMEOUT) {
        char buf[128];
        snprintf(buf, sizeof buf, "op_wait_probe: the wait gave up after %u polls", polls);
        return q3_report_error(Q3_ERR_TIMEOUT, buf);
    }
    if (h != 0) return q3_report_error(Q3_ERR_CUDA, "op_wait_probe: unexpected device status");
    return Q3_OK;
}
