// Host-side TMA tensor-map encoding (driver entry point fetched through the
// runtime, so the library needs no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "common.cuh"

namespace sag {

// Looked up once per process (thread-safe static initialisation); nullptr if
// the driver does not provide it.
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// Row-major [rows, cols] 16-bit tensor, box {64 columns, box_rows}, 128-byte
// swizzle, out-of-range elements read as zero.
inline bool tmap_2d(CUtensorMap *m, const void *base, bool fp16, uint64_t cols, uint64_t rows,
                    uint32_t box_rows) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [d2, d1, d0] 16-bit tensor (d0 contiguous), box {64, 1, box_d2}: picks rows
// strided by d1 * d0 (e.g. the key rows of one KV head in TND layout).
inline bool tmap_3d(CUtensorMap *m, const void *base, bool fp16, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint32_t box_d2) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {64, 1, box_d2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Maps of the query and key tensors of a launch: q as [T1 * n1, d] rows with
// boxes {64, q_box_rows}, k as [T2, n2, d] with boxes {64, 1, k_box}.  With
// the rope split (g.d_rope = 64) q and k hold d_qk - 64 = 128 columns and the
// rope tensors get maps of their own (qr, kr: 64 columns); otherwise qr / kr
// repeat q / k and are never used.
struct QkMaps {
    CUtensorMap q, qr, k, kr;
};
inline bool qk_maps(QkMaps *m, const Geometry &g, const sag_io &io, bool fp16, uint32_t q_box_rows,
                    uint32_t k_box) {
    const uint64_t dq = (uint64_t)(g.d_qk - g.d_rope);
    if (!tmap_2d(&m->q, io.query, fp16, dq, (uint64_t)g.t1 * g.n1, q_box_rows) ||
        !tmap_3d(&m->k, io.key, fp16, dq, g.n2, g.t2, k_box))
        return false;
    if (!g.d_rope) {
        m->qr = m->q;
        m->kr = m->k;
        return true;
    }
    return tmap_2d(&m->qr, io.query_rope, fp16, g.d_rope, (uint64_t)g.t1 * g.n1, q_box_rows) &&
           tmap_3d(&m->kr, io.key_rope, fp16, g.d_rope, g.n2, g.t2, k_box);
}

}  // namespace sag
