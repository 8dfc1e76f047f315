// Allocation-free entry point: the backward with its scratch memory in a
// fixed-size device array that lives in this library's module, so the caller
// passes only inputs and outputs.
//
// Meant for callers that cannot allocate device memory at the point of the
// call: code running under a framework's memory pool that forbids raw
// cudaMalloc, plug-ins handed only tensors by their host, or steps replayed
// where an allocation (and its implicit synchronisation) is not allowed.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr size_t kScratchBytes = SEL_ATTN_GRAD_NOALLOC_MAX_SCRATCH;
constexpr int kMaxDevices = 64;

// One copy per device that loads the library; it stays until process exit.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch per device (the host-side symbol is only a
// stand-in and must never reach a kernel).
void *g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

sag_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return SAG_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SAG_OK;
}

}  // namespace

extern "C" sag_status sel_attn_grad_noalloc(const sag_desc *desc, const void *query, const void *key,
                                            const void *value, const void *attention_out,
                                            const void *attention_out_grad, const float *softmax_max,
                                            const float *softmax_sum, const int32_t *topk_indices,
                                            void *dq, void *dk, void *dv, void *stream) {
    size_t need = 0;
    sag_status st = sel_attn_grad_workspace_size(desc, &need);
    if (st != SAG_OK) return st;
    if (need > kScratchBytes) return SAG_ERR_WORKSPACE;
    // the scratch must belong to the device that runs the stream; the
    // caller's current device is restored on return
    sag::DeviceGuard dg;
    if (!dg.bind(static_cast<cudaStream_t>(stream))) return SAG_ERR_CUDA;
    void *scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != SAG_OK) return st;
    return sel_attn_grad(desc, query, key, value, attention_out, attention_out_grad, softmax_max,
                         softmax_sum, topk_indices, dq, dk, dv, scratch, kScratchBytes, stream);
}

extern "C" sag_status sel_attn_grad_noalloc_query_error(void *stream) {
    sag::DeviceGuard dg;
    if (!dg.bind(static_cast<cudaStream_t>(stream))) return SAG_ERR_CUDA;
    void *scratch = nullptr;
    const sag_status st = scratch_for_current_device(&scratch);
    if (st != SAG_OK) return st;
    return sel_attn_grad_query_error(scratch, stream);
}
