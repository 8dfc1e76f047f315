// Self-test of the device-side failure path every tensor-core kernel of the
// library relies on: a bounded mbarrier wait that runs out records
// SAG_ERR_TIMEOUT in the workspace header and the kernel returns, leaving the
// context usable.  The barrier here is one that no thread and no copy ever
// arrives on, so the wait runs out after `limit_ns`; nothing faults, traps or
// spins without a bound.
#include "kernels.cuh"
#include "tc.cuh"

namespace sag {
namespace {

__global__ void k_wait_timeout(WsHeader *hdr, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phase 0 never completes: the bounded wait gives up and the status is recorded
        if (!tc::mbar_wait(&bar, 0, &abort_flag, limit_ns)) raise_error(&hdr->error, SAG_ERR_TIMEOUT);
        // the wind-down path: nothing was armed, so draining returns at once
        if (!tc::drain_armed(&bar, 0, limit_ns)) raise_error(&hdr->error, SAG_ERR_CUDA);
    }
    __syncthreads();
}

}  // namespace
}  // namespace sag

using namespace sag;

extern "C" sag_status sel_attn_selftest_wait_timeout(void *workspace, uint64_t limit_ns, void *stream) {
    if (!workspace) return SAG_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15) != 0) return SAG_ERR_ALIGN;
    if (limit_ns < 1000 || limit_ns > 4000000000ull) return SAG_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceGuard dg;
    if (!dg.bind(s)) return SAG_ERR_CUDA;
    WsHeader *hdr = static_cast<WsHeader *>(workspace);
    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return SAG_ERR_CUDA;
    k_wait_timeout<<<1, 32, 0, s>>>(hdr, limit_ns);
    return cudaGetLastError() == cudaSuccess ? SAG_OK : SAG_ERR_CUDA;
}
