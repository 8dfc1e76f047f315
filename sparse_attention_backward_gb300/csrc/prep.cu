// Preprocess, index inversion and cast kernels.
//
// Preprocess: Delta[t,h] = sum_d dY[t,h,d] * O[t,h,d] (the rowsum(dY * O) term
// of dS = P * (dP - Delta)) and the log2-domain softmax constant
// lse2 = (softmaxMax + ln softmaxSum) * log2(e), read from lane 0 of the
// [T1, N1, 8] stats ("NsaSelectedAttentionGrad" README, parameters:
// attentionOut, softmaxMax, softmaxSum).
//
// Inversion: topkIndices [T1, N2, count] names, per (token, KV head), the key
// blocks its query rows attend to (README, Gather formula).  The backward
// accumulates dK / dV per key block, so the lists are inverted into
// key-block-major buckets: item = (batch, KV head, block id) -> the
// (token, slot) pairs that selected it, in increasing token order
// (histogram -> exclusive scan -> fill -> per-bucket sort, so the order does
// not depend on atomic timing).
#include "kernels.cuh"

namespace sag {

// ---------------------------------------------------------------------------
// One warp per (t, h) row.  Also zeroes the fp32 dQ accumulator row when
// zero_dq is set (default mode).
template <bool kFp16>
__global__ void __launch_bounds__(256) k_preprocess(Geometry g, const uint16_t *__restrict__ o,
                                                    const uint16_t *__restrict__ dy,
                                                    const float *__restrict__ smax,
                                                    const float *__restrict__ ssum,
                                                    float *__restrict__ delta,
                                                    float *__restrict__ lse2,
                                                    float *__restrict__ dq_acc, int zero_dq) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)g.t1 * g.n1;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp0; r < rows; r += nwarps) {
        const uint16_t *orow = o + r * g.d_v;
        const uint16_t *yrow = dy + r * g.d_v;
        float acc = 0.f;
        // d_v is 128 or 192: lanes take 4 consecutive elements (8 bytes)
        for (int d = lane * 4; d < g.d_v; d += 128) {
            uint2 ov = *reinterpret_cast<const uint2 *>(orow + d);
            uint2 yv = *reinterpret_cast<const uint2 *>(yrow + d);
            const uint16_t *op = reinterpret_cast<const uint16_t *>(&ov);
            const uint16_t *yp = reinterpret_cast<const uint16_t *>(&yv);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc = fmaf(u16_to_f<kFp16>(yp[e]), u16_to_f<kFp16>(op[e]), acc);
        }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
        if (lane == 0) {
            delta[r] = acc;
            const float m = smax[r * 8];
            const float l = ssum[r * 8];
            lse2[r] = (m + logf(l)) * 1.4426950408889634f;
        }
        if (zero_dq) {
            float4 *dst = reinterpret_cast<float4 *>(dq_acc + r * g.d_qk);
            for (int d = lane; d < g.d_qk / 4; d += 32) dst[d] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// ---------------------------------------------------------------------------
// Item of a selection: -1 (reported) when the block id is outside its
// batch's valid blocks, -2 for a padding token (BSND rows past the batch's
// valid length, whose lists are ignored).
__device__ __forceinline__ int64_t item_of(const Geometry &g, const Workspace &ws, int t, int n2, int id) {
    const int b = batch_of(ws.cu_q, g.batch, t);
    if (t >= ws.q_end[b]) return -2;
    if (id < 0 || id >= ws.kv_blocks[b]) return -1;
    const int nblk = (ws.cu_kv[b + 1] - ws.cu_kv[b]) / g.block_size;   // blocks of the (padded) key rows
    return ws.item_base[b] + (int64_t)n2 * nblk + id;
}

__global__ void __launch_bounds__(256) k_histogram(Geometry g, Workspace ws,
                                                   const int32_t *__restrict__ topk) {
    const int64_t n = (int64_t)g.t1 * g.n2 * g.block_count;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / ((int64_t)g.n2 * g.block_count));
        const int n2 = (int)((i / g.block_count) % g.n2);
        const int64_t item = item_of(g, ws, t, n2, __ldg(topk + i));
        if (item == -1) raise_error(&ws.hdr->error, SAG_ERR_INDEX);
        if (item < 0) continue;
        atomicAdd(ws.count + item, 1);
    }
}

// Exclusive scan of count[0..n) into offset[0..n] in three passes:
// per-block sums, a single-block scan of those sums, per-block scans.
constexpr int kScanBlock = 1024;
constexpr int kScanPerThread = 4;
constexpr int kScanTile = kScanBlock * kScanPerThread;

__device__ __forceinline__ int block_exclusive_scan(int v, int *smem_warp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, s);
        if (lane >= s) x += y;
    }
    if (lane == 31) smem_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (blockDim.x >> 5) ? smem_warp[lane] : 0;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, s);
            if (lane >= s) w += y;
        }
        smem_warp[lane] = w;
    }
    __syncthreads();
    const int before = (warp ? smem_warp[warp - 1] : 0) + x - v;
    *total = smem_warp[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kScanBlock) k_scan_partials(const int32_t *__restrict__ in,
                                                              int64_t n, int32_t *__restrict__ part) {
    __shared__ int warp_sums[32];
    const int64_t base = (int64_t)blockIdx.x * kScanTile;
    int v = 0;
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) {
        const int64_t i = base + (int64_t)threadIdx.x * kScanPerThread + e;
        if (i < n) v += in[i];
    }
    int total;
    block_exclusive_scan(v, warp_sums, &total);
    if (threadIdx.x == 0) part[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanBlock) k_scan_tops(int32_t *__restrict__ part, int nparts) {
    __shared__ int warp_sums[32];
    // nparts <= kScanTile (checked on the host): one tile
    int v[kScanPerThread];
    int sum = 0;
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) {
        const int i = threadIdx.x * kScanPerThread + e;
        v[e] = i < nparts ? part[i] : 0;
        sum += v[e];
    }
    int total;
    int run = block_exclusive_scan(sum, warp_sums, &total);
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) {
        const int i = threadIdx.x * kScanPerThread + e;
        if (i < nparts) part[i] = run;
        run += v[e];
    }
}

__global__ void __launch_bounds__(kScanBlock) k_scan_apply(const int32_t *__restrict__ in, int64_t n,
                                                           const int32_t *__restrict__ part,
                                                           int32_t *__restrict__ out) {
    __shared__ int warp_sums[32];
    const int64_t base = (int64_t)blockIdx.x * kScanTile;
    int v[kScanPerThread];
    int sum = 0;
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) {
        const int64_t i = base + (int64_t)threadIdx.x * kScanPerThread + e;
        v[e] = i < n ? in[i] : 0;
        sum += v[e];
    }
    int total;
    int run = block_exclusive_scan(sum, warp_sums, &total) + part[blockIdx.x];
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) {
        const int64_t i = base + (int64_t)threadIdx.x * kScanPerThread + e;
        if (i < n) out[i] = run;
        run += v[e];
    }
    // offset[n] = grand total, written by the block holding element n-1
    if (base <= n - 1 && n - 1 < base + kScanTile && threadIdx.x == 0) {
        int grand = part[blockIdx.x] + total;
        out[n] = grand;
    }
}

__global__ void __launch_bounds__(256) k_fill(Geometry g, Workspace ws,
                                              const int32_t *__restrict__ topk) {
    const int64_t n = (int64_t)g.t1 * g.n2 * g.block_count;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / ((int64_t)g.n2 * g.block_count));
        const int n2 = (int)((i / g.block_count) % g.n2);
        const int slot = (int)(i % g.block_count);
        const int64_t item = item_of(g, ws, t, n2, __ldg(topk + i));
        if (item < 0) continue;
        const int pos = ws.offset[item] + atomicAdd(ws.cursor + item, 1);
        ws.entries[pos] = t * g.block_count + slot;
    }
}

// Sort each bucket ascending (token-major order), so that the order of the
// entries does not depend on the timing of the fill's atomics.  Needed where
// the order matters: the deterministic mode (fixed accumulation order), token
// chunks and token windows (binary searches by token); the default mode takes
// the buckets as filled.  The network
// is bitonic in its all-ascending form (the first step of every merge pairs
// i with its mirror i ^ (k - 1), the later ones pair i with i ^ j), which
// lets a bucket of n entries be padded virtually to the next power of two
// with +infinity: such a pad never moves below index n, so pairs whose upper
// index is >= n are skipped and nothing is written beyond the bucket.
// Buckets of up to kSortCap entries are sorted whole in shared memory.
// Larger ones (e.g. a block that every query of a long batch selects) are
// sorted in place by the same CTA: every kSortCap chunk in shared memory, then
// the merge steps whose stride spans chunks as passes over global memory, and
// after each such step the short strides again chunk by chunk in shared memory.
// With token windows, each item then records where every window of its batch
// starts inside its sorted bucket.
constexpr int kSortCap = 16384;

// The steps of stage k whose strides are < kSortCap, on one chunk of the
// bucket held in shared memory (keys[0 .. len) real, the rest +infinity).
// Each thread takes compare-exchange pairs q (lower index i, upper l), p2 / 2
// of them per step: i keeps bit j clear (l = i + j), or for the mirror step i
// is in the lower half of its k-block (l = i ^ (k - 1)).
__device__ __forceinline__ void sort_steps_smem(int32_t *keys, int p2, int k_lo, int k_hi, bool mirror_first) {
    for (int k = k_lo; k <= k_hi; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            const bool mirror = mirror_first && j == (k >> 1);
            const int lj = __ffs(j) - 1;   // j = 2^lj (for the mirror step also k / 2)
            for (int q = threadIdx.x; q < (p2 >> 1); q += blockDim.x) {
                const int i = ((q >> lj) << (lj + 1)) + (q & (j - 1));
                const int l = mirror ? (i ^ (k - 1)) : (i + j);
                const int32_t x = keys[i], y = keys[l];
                if (x > y) { keys[i] = y; keys[l] = x; }
            }
            __syncthreads();
        }
    }
}

// Load chunk c of a (length n) into keys, padding with +infinity.
__device__ __forceinline__ void chunk_load(int32_t *keys, const int32_t *a, int n, int c) {
    for (int i = threadIdx.x; i < kSortCap; i += blockDim.x) {
        const int gi = c * kSortCap + i;
        keys[i] = gi < n ? a[gi] : INT32_MAX;
    }
    __syncthreads();
}
__device__ __forceinline__ void chunk_store(const int32_t *keys, int32_t *a, int n, int c) {
    for (int i = threadIdx.x; i < kSortCap; i += blockDim.x) {
        const int gi = c * kSortCap + i;
        if (gi < n) a[gi] = keys[i];
    }
    __syncthreads();
}

__device__ void sort_large_bucket(int32_t *a, int n, int32_t *keys) {
    int p2 = kSortCap;
    while (p2 < n) p2 <<= 1;
    const int nchunks = (n + kSortCap - 1) / kSortCap;
    // stages k = 2 .. kSortCap: each chunk on its own
    for (int c = 0; c < nchunks; ++c) {
        chunk_load(keys, a, n, c);
        sort_steps_smem(keys, kSortCap, 2, kSortCap, true);
        chunk_store(keys, a, n, c);
    }
    for (int k = 2 * kSortCap; k <= p2; k <<= 1) {
        // strides >= kSortCap in global memory (mirror step first)
        for (int j = k >> 1; j >= kSortCap; j >>= 1) {
            const bool mirror = j == (k >> 1);
            for (int i = threadIdx.x; i < p2; i += blockDim.x) {
                const int l = mirror ? (i ^ (k - 1)) : (i ^ j);
                if (l > i && l < n) {
                    const int32_t x = a[i], y = a[l];
                    if (x > y) { a[i] = y; a[l] = x; }
                }
            }
            __syncthreads();
        }
        // strides < kSortCap chunk by chunk (no mirror step: plain half-cleaners)
        for (int c = 0; c < nchunks; ++c) {
            chunk_load(keys, a, n, c);
            for (int j = kSortCap >> 1; j > 0; j >>= 1) {
                const int lj = __ffs(j) - 1;
                for (int q = threadIdx.x; q < (kSortCap >> 1); q += blockDim.x) {
                    const int i = ((q >> lj) << (lj + 1)) + (q & (j - 1)), l = i + j;
                    const int32_t x = keys[i], y = keys[l];
                    if (x > y) { keys[i] = y; keys[l] = x; }
                }
                __syncthreads();
            }
            chunk_store(keys, a, n, c);
        }
    }
}

__global__ void __launch_bounds__(512) k_sort_buckets(Geometry g, Workspace ws) {
    extern __shared__ int32_t keys[];   // kSortCap entries
    for (int64_t item = blockIdx.x; item < g.n_items; item += gridDim.x) {
        const int off = ws.offset[item];
        const int n = ws.offset[item + 1] - off;
        int32_t *a = ws.entries + off;
        const bool in_smem = n <= kSortCap;
        if (n > 1) {
            if (!in_smem) {
                sort_large_bucket(a, n, keys);
            } else {
                int p2 = 1;
                while (p2 < n) p2 <<= 1;
                for (int i = threadIdx.x; i < p2; i += blockDim.x) keys[i] = i < n ? a[i] : INT32_MAX;
                __syncthreads();
                sort_steps_smem(keys, p2, 2, p2, true);
                for (int i = threadIdx.x; i < n; i += blockDim.x) a[i] = keys[i];
            }
        } else if (n == 1) {
            if (threadIdx.x == 0) keys[0] = a[0];
        }
        __syncthreads();
        if (g.windowed) {
            const int b = batch_of_item(ws.item_base, g.batch, item);
            const int nwin = n_windows(g, ws.cu_q, b);
            const int32_t *src = in_smem ? keys : a;
            int32_t *tab = ws.wtab + ws.wtab_base[b] + (item - ws.item_base[b]) * (int64_t)(nwin + 1);
            for (int w = threadIdx.x; w <= nwin; w += blockDim.x) {
                const int t0 = ws.cu_q[b] + w * g.window;   // first token of window w
                int lo = 0, hi = n;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (src[mid] / g.block_count < t0) lo = mid + 1; else hi = mid;
                }
                tab[w] = off + lo;
            }
        }
        __syncthreads();
    }
}

// dQ = scale * the fp32 accumulator, rounded to 16 bits; with the rope split
// the columns from d_qk - d_rope on go to dq_rope (a group of 4 never straddles
// the boundary: both widths are multiples of 4).
template <bool kFp16>
__global__ void __launch_bounds__(256) k_cast_dq(Geometry g, const float *__restrict__ in, uint16_t *__restrict__ out,
                                                 uint16_t *__restrict__ out_rope, int64_t n4) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = reinterpret_cast<const float4 *>(in)[i];
        ushort4 o;
        o.x = f_to_u16<kFp16>(v.x * g.scale);
        o.y = f_to_u16<kFp16>(v.y * g.scale);
        o.z = f_to_u16<kFp16>(v.z * g.scale);
        o.w = f_to_u16<kFp16>(v.w * g.scale);
        const int64_t row = (i * 4) / g.d_qk;
        const int col = (int)((i * 4) % g.d_qk);
        *reinterpret_cast<ushort4 *>(split_col(out, out_rope, row, col, g.d_qk, g.d_rope)) = o;
    }
}

// ---------------------------------------------------------------------------
// Fixed-order dQ from per-slot partials.  The main kernel stored, for every
// (query row, selection slot, key tile of the block), the fp32 partial
// dS_tile K_tile of that row; here one warp per row of the token chunk sums
// them in list order (slot, then tile) and writes scale * sum in the dtype
// (dQ = dS K / sqrt(d), README function description).  Slots whose id is
// empty, out of range or on a padding token were never stored; they are
// skipped by the test the inversion applies.  Eight slots are loaded before
// they are added, always in the same order.
template <bool kFp16, int DQK>
__global__ void __launch_bounds__(256) k_dq_slot_sum(Geometry g, Workspace ws, const int32_t *__restrict__ topk,
                                                     uint16_t *__restrict__ dq, uint16_t *__restrict__ dq_rope) {
    constexpr int V4 = DQK / 4;                 // float4 per row: 32 or 48
    constexpr int PER = (V4 + 31) / 32;         // per lane: 1 or 2
    constexpr int U = 8;                        // slots in flight
    const int lane = threadIdx.x & 31;
    const int nsl = g.block_count * g.halves;
    const int64_t nrows = (int64_t)(g.tok_hi - g.tok_lo) * g.n1;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = (((int64_t)blockIdx.x * blockDim.x) >> 5) + (threadIdx.x >> 5); r < nrows; r += warps) {
        const int t = g.tok_lo + (int)(r / g.n1), h = (int)(r % g.n1);
        const int b = batch_of(ws.cu_q, g.batch, t);
        const int nblk = t < ws.q_end[b] ? ws.kv_blocks[b] : 0;
        const int32_t *ids = topk + ((int64_t)t * g.n2 + h / g.group) * g.block_count;
        const float4 *part = reinterpret_cast<const float4 *>(ws.dq_part) + r * nsl * V4;
        float4 acc[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < nsl; j0 += U) {
            float4 v[U][PER];
            bool use[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u;
                int id = -1;
                if (j < nsl) id = __ldg(ids + j / g.halves);
                use[u] = id >= 0 && id < nblk;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    const int c = lane + 32 * q;
                    v[u][q] = (use[u] && c < V4) ? __ldcs(part + (int64_t)j * V4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (use[u])
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        acc[q].x += v[u][q].x;
                        acc[q].y += v[u][q].y;
                        acc[q].z += v[u][q].z;
                        acc[q].w += v[u][q].w;
                    }
        }
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int c = lane + 32 * q;
            if (c >= V4) continue;
            ushort4 o;
            o.x = f_to_u16<kFp16>(acc[q].x * g.scale);
            o.y = f_to_u16<kFp16>(acc[q].y * g.scale);
            o.z = f_to_u16<kFp16>(acc[q].z * g.scale);
            o.w = f_to_u16<kFp16>(acc[q].w * g.scale);
            *reinterpret_cast<ushort4 *>(split_col(dq, dq_rope, (int64_t)t * g.n1 + h, 4 * c, DQK, g.d_rope)) = o;
        }
    }
}

// ---------------------------------------------------------------------------
// Host launchers.
static int grid_for(int64_t work, int per_block, int max_blocks) {
    int64_t b = (work + per_block - 1) / per_block;
    if (b < 1) b = 1;
    if (b > max_blocks) b = max_blocks;
    return (int)b;
}

cudaError_t launch_preprocess(const Geometry &g, const Workspace &ws, const void *o, const void *dy,
                              const float *smax, const float *ssum, bool fp16, bool zero_dq,
                              cudaStream_t s, int num_sms) {
    const int64_t rows = (int64_t)g.t1 * g.n1;
    const int grid = grid_for(rows, 8, num_sms * 16);
    if (rows == 0) return cudaSuccess;
    if (fp16)
        k_preprocess<true><<<grid, 256, 0, s>>>(g, (const uint16_t *)o, (const uint16_t *)dy, smax, ssum,
                                                ws.delta, ws.lse2, ws.dq_acc, zero_dq);
    else
        k_preprocess<false><<<grid, 256, 0, s>>>(g, (const uint16_t *)o, (const uint16_t *)dy, smax, ssum,
                                                 ws.delta, ws.lse2, ws.dq_acc, zero_dq);
    return cudaGetLastError();
}

int scan_parts(int64_t n_items) { return (int)((n_items + kScanTile - 1) / kScanTile); }
int64_t max_scannable_items() { return (int64_t)kScanTile * kScanTile; }

cudaError_t launch_inversion(const Geometry &g, const Workspace &ws, const int32_t *topk, bool sorted, cudaStream_t s,
                             int num_sms) {
    const int64_t sel = (int64_t)g.t1 * g.n2 * g.block_count;
    if (sel > 0) {
        k_histogram<<<grid_for(sel, 256, num_sms * 8), 256, 0, s>>>(g, ws, topk);
    }
    const int parts = scan_parts(g.n_items);
    k_scan_partials<<<parts, kScanBlock, 0, s>>>(ws.count, g.n_items, ws.scan_part);
    k_scan_tops<<<1, kScanBlock, 0, s>>>(ws.scan_part, parts);
    k_scan_apply<<<parts, kScanBlock, 0, s>>>(ws.count, g.n_items, ws.scan_part, ws.offset);
    if (sel > 0) {
        k_fill<<<grid_for(sel, 256, num_sms * 8), 256, 0, s>>>(g, ws, topk);
        if (sorted) {
            cudaFuncSetAttribute(k_sort_buckets, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kSortCap * sizeof(int32_t)));
            k_sort_buckets<<<grid_for(g.n_items, 1, num_sms * 4), 512, kSortCap * sizeof(int32_t), s>>>(g, ws);
        }
    }
    return cudaGetLastError();
}

cudaError_t launch_cast_dq(const Geometry &g, const float *dq_acc, void *dq, void *dq_rope, bool fp16,
                           cudaStream_t s, int num_sms) {
    const int64_t n4 = (int64_t)g.t1 * g.n1 * g.d_qk / 4;
    if (n4 == 0) return cudaSuccess;
    const int grid = grid_for(n4, 256, num_sms * 8);
    if (fp16) k_cast_dq<true><<<grid, 256, 0, s>>>(g, dq_acc, (uint16_t *)dq, (uint16_t *)dq_rope, n4);
    else k_cast_dq<false><<<grid, 256, 0, s>>>(g, dq_acc, (uint16_t *)dq, (uint16_t *)dq_rope, n4);
    return cudaGetLastError();
}

template <bool kFp16, int DQK>
static cudaError_t launch_dq_slots_t(const Geometry &g, const Workspace &ws, const sag_io &io, cudaStream_t s,
                                     int num_sms) {
    const int64_t rows = (int64_t)(g.tok_hi - g.tok_lo) * g.n1;
    if (rows == 0) return cudaSuccess;
    const int grid = grid_for(rows, 8, num_sms * 8);
    k_dq_slot_sum<kFp16, DQK><<<grid, 256, 0, s>>>(g, ws, io.topk_indices, (uint16_t *)io.dq, (uint16_t *)io.dq_rope);
    return cudaGetLastError();
}

cudaError_t launch_dq_slots(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, cudaStream_t s,
                            int num_sms) {
    if (g.d_qk != 128 && g.d_qk != 192) return cudaErrorInvalidValue;
    if (fp16)
        return g.d_qk == 192 ? launch_dq_slots_t<true, 192>(g, ws, io, s, num_sms)
                             : launch_dq_slots_t<true, 128>(g, ws, io, s, num_sms);
    return g.d_qk == 192 ? launch_dq_slots_t<false, 192>(g, ws, io, s, num_sms)
                         : launch_dq_slots_t<false, 128>(g, ws, io, s, num_sms);
}

}  // namespace sag
