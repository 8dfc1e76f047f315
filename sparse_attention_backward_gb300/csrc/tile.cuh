// Pieces shared by the tensor-core kernels that walk key tiles (backward and
// forward): the work-unit decode over the inverted index, the CTA shape, and
// small numeric / layout helpers.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace sag {
namespace {

constexpr int kThreads = 320;       // warp 0 TMA, warp 1 MMA, warps 2-5 softmax, warps 6-9 epilogue
constexpr int kRows = 128;          // query rows per tile (MMA M)
constexpr uint64_t kWaitNs = 2000000000ull;

struct KeyTile {
    int b, n2;
    int64_t key0;       // first key row
    int koff;           // offset of the tile inside its block
    int64_t item;
    int e0, ntok;       // bucket entries [e0, e0 + ntok) of this launch's token range
    int ntiles;
};

// Work unit u -> key tile and its bucket entries.  Windowed: units of batch b
// are ordered (KV head, window, block, half); the bucket range of a window
// comes from the window table.  Otherwise u = item * halves + half and the
// range is this launch's token chunk of the bucket.
__device__ __forceinline__ KeyTile decode(const Geometry &g, const Workspace &ws, int64_t u, int nk, int tpt) {
    KeyTile kt;
    const int halves = g.halves;
    int half, kb, nblk;
    if (g.windowed) {
        kt.b = batch_of_item(ws.unit_base, g.batch, u);
        nblk = (ws.cu_kv[kt.b + 1] - ws.cu_kv[kt.b]) / g.block_size;
        const int nwin = n_windows(g, ws.cu_q, kt.b);
        const int64_t local = u - ws.unit_base[kt.b];
        const int64_t per_head = (int64_t)nwin * nblk * halves;
        kt.n2 = (int)(local / per_head);
        const int64_t rem = local % per_head;
        const int w = (int)(rem / (nblk * halves));
        const int rem2 = (int)(rem % (nblk * halves));
        kb = rem2 / halves;
        half = rem2 % halves;
        kt.item = ws.item_base[kt.b] + (int64_t)kt.n2 * nblk + kb;
        const int32_t *tab = ws.wtab + ws.wtab_base[kt.b] + (kt.item - ws.item_base[kt.b]) * (int64_t)(nwin + 1);
        kt.e0 = tab[w];
        kt.ntok = tab[w + 1] - kt.e0;
    } else {
        kt.item = u / halves;
        half = (int)(u % halves);
        kt.b = batch_of_item(ws.item_base, g.batch, kt.item);
        nblk = (ws.cu_kv[kt.b + 1] - ws.cu_kv[kt.b]) / g.block_size;
        const int64_t local = kt.item - ws.item_base[kt.b];
        kt.n2 = (int)(local / nblk);
        kb = (int)(local % nblk);
        const int e_end = ws.offset[kt.item + 1];
        if (g.tok_lo == 0 && g.tok_hi == g.t1) {
            kt.e0 = ws.offset[kt.item];
            kt.ntok = e_end - kt.e0;
        } else {
            kt.e0 = lower_bound_token(ws.entries, ws.offset[kt.item], e_end, g.tok_lo, g.block_count);
            kt.ntok = lower_bound_token(ws.entries, kt.e0, e_end, g.tok_hi, g.block_count) - kt.e0;
        }
    }
    kt.koff = half * nk;
    kt.key0 = ws.cu_kv[kt.b] + (int64_t)kb * g.block_size + kt.koff;
    kt.ntiles = (kt.ntok + tpt - 1) / tpt;
    return kt;
}

// Dynamic work distribution.  Warp 0 of a CTA takes the next work unit from
// a launch-wide ticket counter (atomic add) and publishes it in a small shared
// ring; every other role reads the units from the ring in the same order.  A
// unit index >= n_units ends the sequence.  The functions are warp-collective
// and return -1 when a bounded wait ran out.
constexpr int kURing = 4;
struct UnitRing {
    int64_t *slot;          // [kURing] in shared memory
    uint64_t *full;         // [kURing] mbarriers, one arrival (the producer)
    uint64_t *empty;        // [kURing] mbarriers, one arrival per consumer warp
};

__device__ __forceinline__ int64_t ring_take(const UnitRing &r, unsigned long long *counter, int k,
                                             volatile int *abort, int lane) {
    const int q = k % kURing;
    if (k >= kURing &&
        !__all_sync(0xffffffffu, tc::mbar_wait(&r.empty[q], ((k / kURing) - 1) & 1, abort, kWaitNs)))
        return -1;
    int64_t ti = 0;
    if (lane == 0) {
        ti = (int64_t)atomicAdd(counter, 1ull);
        r.slot[q] = ti;
        tc::mbar_arrive(&r.full[q]);
    }
    return __shfl_sync(0xffffffffu, ti, 0);
}

__device__ __forceinline__ int64_t ring_read(const UnitRing &r, int k, volatile int *abort, int lane) {
    const int q = k % kURing;
    if (!__all_sync(0xffffffffu, tc::mbar_wait(&r.full[q], (k / kURing) & 1, abort, kWaitNs))) return -1;
    const int64_t ti = *reinterpret_cast<volatile int64_t *>(&r.slot[q]);
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&r.empty[q]);
    return ti;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// a in the low half, b in the high half, both rounded to nearest even (one
// paired conversion instead of two scalar ones)
template <bool kFp16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (kFp16) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// address of 16-byte chunk c of row r in a 128-byte-swizzled [rows x 128 B] tile
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace
}  // namespace sag
