// Launchers of the library's kernels (host side).
#pragma once

#include "common.cuh"

namespace sag {

// Makes the device that owns a stream current for the length of one library
// call and gives the calling thread its previous current device back when it
// goes out of scope (the legacy default stream, NULL, keeps the current one).
class DeviceGuard {
public:
    DeviceGuard() = default;
    DeviceGuard(const DeviceGuard &) = delete;
    DeviceGuard &operator=(const DeviceGuard &) = delete;
    bool bind(cudaStream_t s);
    ~DeviceGuard();

private:
    int saved_ = -1;
};

cudaError_t launch_preprocess(const Geometry &g, const Workspace &ws, const void *o, const void *dy,
                              const float *smax, const float *ssum, bool fp16, bool zero_dq,
                              cudaStream_t s, int num_sms);
// topkIndices -> per key block the (token, slot) pairs naming it; `sorted`
// orders each bucket by token (the fill's own order depends on atomic timing)
cudaError_t launch_inversion(const Geometry &g, const Workspace &ws, const int32_t *topk, bool sorted, cudaStream_t s,
                             int num_sms);
// scale * dq_acc -> dq (and dq_rope: columns d_qk - d_rope .. d_qk - 1)
cudaError_t launch_cast_dq(const Geometry &g, const float *dq_acc, void *dq, void *dq_rope, bool fp16,
                           cudaStream_t s, int num_sms);
int scan_parts(int64_t n_items);
int64_t max_scannable_items();

// CUDA-core key-block-major backward (any supported shape without the rope split).
cudaError_t launch_bwd_simt(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16,
                            bool deterministic, cudaStream_t s, int num_sms);
// Tensor-core (tcgen05) key-block-major backward: d_v == 128, d_qk in
// {128, 192}, block size in {16, 32, 48, 64, 128}.
bool bwd_tc_supported(const Geometry &g);
cudaError_t launch_bwd_tc(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, bool deterministic,
                          cudaStream_t s, int num_sms);
// The same backward with the softmax split in two phases (bwd_tc_split.cu),
// preferred for small query groups.
bool bwd_split_preferred(const Geometry &g);
cudaError_t launch_bwd_tc_split(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16,
                                bool deterministic, cudaStream_t s, int num_sms);
// dK/dV from the fp32 accumulator after the last token chunk.
cudaError_t launch_cast_dkv(const Geometry &g, const Workspace &ws, void *dk, void *dk_rope, void *dv, bool fp16,
                            cudaStream_t s, int num_sms);
// Tensor-core dQ from the stored dS, fixed order (deterministic mode):
// d_qk in {128, 192}, block size 64 or 128.
bool dq_tc_supported(const Geometry &g);
cudaError_t launch_dq_tc(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, cudaStream_t s,
                         int num_sms);
// Forward (tensor cores, same shapes as the backward's tensor-core kernel):
// row state init, pass 1 (row maxima) / pass 2 (row sums and O), finalize.
bool fwd_tc_supported(const Geometry &g);
cudaError_t launch_fwd_init(const Geometry &g, const Workspace &ws, cudaStream_t s, int num_sms);
cudaError_t launch_fwd_tc(const Geometry &g, const Workspace &ws, const sag_io &io, int pass, bool fp16,
                          cudaStream_t s, int num_sms);
cudaError_t launch_fwd_finalize(const Geometry &g, const Workspace &ws, void *o, float *smax, float *ssum, bool fp16,
                                cudaStream_t s, int num_sms);
// dQ from the stored dS, fixed order (deterministic mode).
cudaError_t launch_dq_from_ds(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, cudaStream_t s,
                              int num_sms);
// Fixed-order dQ from the per-slot fp32 partials of one token chunk
// (Geometry::dq_slots): dQ = scale * sum over the row's selections in list
// order, cast to the dtype (prep.cu).
cudaError_t launch_dq_slots(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, cudaStream_t s,
                            int num_sms);

// Lightning-indexer backward (tensor cores): head dim 128, G = n1 / n2 <= 64.
// Geometry: t1 / t2 rows, n1, n2, group, block_count = topk; Workspace: hdr,
// cu_q / cu_kv row starts, q_end, kv_blocks = valid key rows of each batch,
// dq_acc = fp32 dK accumulator [t2 * n2, 128], dkv_acc = fp32 dW accumulator.
bool lig_tc_supported(const Geometry &g);
cudaError_t launch_lig(const Geometry &g, const Workspace &ws, const sli_io &io, bool fp16, cudaStream_t s,
                       int num_sms);

// Element (row, col) of a [rows, d_qk] gradient whose columns from d_qk -
// d_rope on live in a separate [rows, d_rope] tensor (the rope split).
__device__ __forceinline__ uint16_t *split_col(uint16_t *main, uint16_t *rope, int64_t row, int col, int d_qk,
                                               int d_rope) {
    const int d_main = d_qk - d_rope;
    return col < d_main ? main + row * d_main + col : rope + row * d_rope + (col - d_main);
}

}  // namespace sag
