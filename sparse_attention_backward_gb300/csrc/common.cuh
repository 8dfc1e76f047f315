// Shared device/host definitions of the selected-attention backward library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/selattn.h"

namespace sag {

// ---------------------------------------------------------------------------
// 16-bit element access.  kFp16 selects half, otherwise bfloat16.
template <bool kFp16> struct Elem;
template <> struct Elem<false> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float to_f(T x) { return __bfloat162float(x); }
    static __device__ __forceinline__ T from_f(float x) { return __float2bfloat16_rn(x); }
    static __device__ __forceinline__ float2 to_f2(__nv_bfloat162 x) { return __bfloat1622float2(x); }
};
template <> struct Elem<true> {
    using T = __half;
    static __device__ __forceinline__ float to_f(T x) { return __half2float(x); }
    static __device__ __forceinline__ T from_f(float x) { return __float2half_rn(x); }
    static __device__ __forceinline__ float2 to_f2(__half2 x) { return __half22float2(x); }
};

// raw 16-bit -> float
template <bool kFp16>
__device__ __forceinline__ float u16_to_f(uint16_t bits) {
    if constexpr (kFp16) return __half2float(__ushort_as_half(bits));
    else return __bfloat162float(__ushort_as_bfloat16(bits));
}
template <bool kFp16>
__device__ __forceinline__ uint16_t f_to_u16(float x) {
    if constexpr (kFp16) return __half_as_ushort(__float2half_rn(x));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------------------
// Device-recorded status: the first non-zero code wins.
__device__ __forceinline__ void raise_error(int *flag, int code) { atomicCAS(flag, 0, code); }

// ---------------------------------------------------------------------------
// Problem geometry shared by every kernel (passed by value).
struct Geometry {
    int32_t batch;
    int32_t t1, t2;
    int32_t n1, n2, group;
    int32_t d_qk, d_v;
    int32_t block_size, block_count;
    int64_t n_items;          // sum_b n2 * (S2_b / block_size)
    float scale;              // scaleValue as fp32
    float scale_log2;         // scale * log2(e): exp(scale*x - lse) = exp2(x*scale_log2 - lse2)
    int32_t tok_lo, tok_hi;   // query tokens handled by this launch (a chunk, or [0, T1))
    int32_t chunked;          // 1: dK/dV carried across launches in the fp32 accumulator
    // Token windows (tensor-core default mode): the work of each (batch, KV
    // head) is split into windows of `window` query tokens, processed window
    // by window, so that one window's dQ accumulator rows stay in L2.  dK/dV
    // then arrive as per-window partials, reduced into the fp32 accumulator.
    int32_t windowed;         // 1: units are (batch, KV head, window, key tile)
    int32_t window;           // tokens per window
    int32_t halves;           // key tiles per block (block_size / key tile)
    int32_t d_rope;           // columns [d_qk - d_rope, d_qk) of q / k live in the rope tensors
    int32_t dq_slots;         // 1: fixed-order dQ from fp32 partials per (row, slot, key tile)
    int64_t n_units;          // work units of the main kernel
};

// Workspace header (first 256 bytes).
struct WsHeader {
    int32_t error;            // sag_status recorded by the device
    int32_t pad0;
    unsigned long long work_counter;   // next work unit of a dynamically scheduled launch
    int32_t pad[60];
};

// Device pointers carved out of the caller's workspace.
struct Workspace {
    WsHeader *hdr;
    int32_t *cu_q;            // [B+1] first query row of each batch (TND: cu_seqlens_q; BSND: b * s1_max)
    int32_t *cu_kv;           // [B+1] first key row of each batch (TND: cu_seqlens_kv; BSND: b * s2_max)
    int32_t *q_end;           // [B]   end of the valid query rows of each batch
    int32_t *kv_blocks;       // [B]   valid key blocks of each batch (ids must be below)
    int64_t *item_base;       // [B+1] first item id of each batch
    int32_t *count;           // [n_items + 1]  selections naming each item
    int32_t *offset;          // [n_items + 1]  exclusive prefix of count
    int32_t *cursor;          // [n_items]      fill cursors
    int32_t *scan_part;       // [scan blocks]  partial sums of the scan
    int32_t *entries;         // [T1 * n2 * count] (token * block_count + slot), bucketed by item
    float *delta;             // [T1 * n1]  rowsum(dY * O)
    float *lse2;              // [T1 * n1]  (max + ln sum) * log2(e)
    float *dq_acc;            // [T1 * n1 * d_qk] fp32 dQ accumulator (default mode)
    uint16_t *ds;             // [chunk tokens * n2 * count * G * bs] dS in the input dtype (deterministic)
    float *dq_part;           // [chunk tokens * n1 * count * halves * d_qk] fp32 dQ partials (dq_slots)
    float *dkv_acc;           // [T2 * n2 * (d_qk + d_v)] fp32 dK|dV carried across chunks / windows
    int64_t *unit_base;       // [B+1] first work unit of each batch (windowed)
    int64_t *wtab_base;       // [B+1] first window-table entry of each batch (windowed)
    int32_t *wtab;            // per item: nwin_b + 1 bucket positions, window starts (windowed)
};

// Windows of batch b: ceil(S1_b / window).
__device__ __forceinline__ int n_windows(const Geometry &g, const int32_t *cu_q, int b) {
    const int s1 = cu_q[b + 1] - cu_q[b];
    return (s1 + g.window - 1) / g.window;
}

// First entry of a sorted bucket [lo, hi) whose token is >= t.
__device__ __forceinline__ int lower_bound_token(const int32_t *e, int lo, int hi, int t, int cnt) {
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (e[mid] / cnt < t) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Batch of a query token (binary search over cu_q, which has B+1 entries).
__device__ __forceinline__ int batch_of(const int32_t *cu_q, int batch, int t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Batch of an item (binary search over item_base).
__device__ __forceinline__ int batch_of_item(const int64_t *item_base, int batch, int64_t item) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(item_base + mid) <= item) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace sag
