// Lightning-indexer backward on tensor cores ("aclnnLightningIndexerGrad",
// formula section):
//     S  = Relu(Matmul(Query, Gather(Key, Indices)))
//     Y  = Dy * Weights,  R = ReluGrad(Y, S) = Y where S > 0, else 0
//     dW = Reduce(S * dy),  dQ = Matmul(R, Gather(Key, Indices)),
//     dK = ScatterAdd(Matmul(R^T, Q), Indices)
// for query head h of key head n2 = h / G:  S[t,h,j] = relu(<q[t,h], k[idx[t,n2,j]]>),
// R[t,h,j] = dy[t,n2,j] * w[t,h] * [S > 0].
//
// Work unit: one (query token t, key head n2) and its topk selections, taken
// in chunks of 128 gathered key rows.  Per chunk (heads padded to 64):
//     S^T  = Kc Q^T       (M = 128 keys, N = 64 heads, K = d)     -> TMEM
//     R    from S^T, dy, w  (CUDA cores, thread = key = TMEM lane) -> shared
//     dQ^T += Kc^T R      (M = d dims, N = 64 heads, K = 128 keys) TMEM, per unit
//     dKc  = R Q          (M = 128 keys, N = d dims, K = 64 heads)   -> TMEM
// dKc is scatter-added (fp32 reductions) into a workspace accumulator at the
// gathered key rows; dQ is stored once per unit (a unit owns its rows); dW is
// reduced over the chunk's keys with warp butterflies.
//
// Warp roles (320 threads): 0 TMA producer (query rows, key rows by
// tile::gather4, the unit's weights), 1 MMA issuer and TMEM owner, 2-5 relu /
// dW (thread = key; dW partials added into an fp32 row with atomics),
// 6-9 epilogue (dK reductions, dQ stores).  Every wait is bounded and there
// is no block-level barrier between the roles.
#include "kernels.cuh"
#include "tc.cuh"
#include "tile.cuh"
#include "tmap.cuh"

namespace sag {
namespace {

constexpr int kLiD = 128;            // head dim
constexpr int kLiChunk = 128;        // gathered keys per chunk (MMA M)
constexpr int kLiHeads = 64;         // heads per unit, padded (MMA N)
// warps: 0 lead producer, 1 MMA, 2-5 relu / dW, 6-9 epilogue, 10 second key
// loader (a warp issues one tile::gather4 about every 66 cycles: one warp
// alone would spend ~4k cycles per chunk on the key rows)
constexpr int kLiLoader2 = 10;
constexpr int kLiThreads = (kLiLoader2 + 1) * 32;

// TMEM columns: S^T stages, dK stages, dQ^T buffers (512 allocated)
constexpr uint32_t kLiColS = 0, kLiColDK = 128, kLiColDQ = 384;

constexpr int kLiKStages = 3;       // gathered key tiles in flight

struct LiSmem {
    static constexpr int K_STAGE = 2 * kLiChunk * 128;     // 2 chunks of 64 dims x 128 rows
    static constexpr int Q_STAGE = 2 * kLiHeads * 128;     // 2 chunks of 64 dims x 64 head rows
    static constexpr int R_STAGE = kLiChunk * 128;         // 128 key rows x 64 heads (bf16)
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = OFF_K + kLiKStages * K_STAGE;
    static constexpr int OFF_R = OFF_Q + 2 * Q_STAGE;
    static constexpr int OFF_STG = OFF_R + 2 * R_STAGE;      // 4 epilogue warps x 4 KB
    static constexpr int OFF_W = OFF_STG + 16384;            // 2 x 64 weights (fp32), by query stage
    static constexpr int OFF_BAR = OFF_W + 2 * kLiHeads * 4;
    static constexpr int TOTAL = OFF_BAR + 256 + 1024;
};

enum LiBar {
    L_Q_FULL0 = 0, L_Q_FULL1, L_Q_EMPTY0, L_Q_EMPTY1, L_K_FULL0, L_K_EMPTY0 = L_K_FULL0 + kLiKStages,
    L_S_FULL0 = L_K_EMPTY0 + kLiKStages, L_S_FULL1, L_R_FULL0, L_R_FULL1, L_DK_FULL0, L_DK_FULL1, L_DK_FREE0, L_DK_FREE1,
    L_DQ_FULL0, L_DQ_FULL1, L_DQ_FREE0, L_DQ_FREE1, L_DRAIN, L_COUNT
};

struct LiArgs {
    Geometry g;            // batch, t1, t2, n1, n2, group; block_count = topk
    Workspace ws;          // hdr, cu_q / cu_kv (row starts), q_end, kv_blocks = valid key rows,
                           // dq_acc = fp32 dK accumulator, dkv_acc = fp32 dW accumulator
    const int32_t *idx;    // [T1, n2, topk]
    const float *dy;       // [T1, n2, topk]
    const uint16_t *w;     // [T1, n1]
    uint16_t *dq;          // [T1, n1, d]
    int64_t n_units;       // T1 * n2
    int nchunks;           // ceil(topk / 128)
};

// A unit's view of its selections: index list, dy row, the batch's valid key
// rows and first key-map row.
struct LiUnit {
    const int32_t *idx;    // [topk]
    const float *dy;       // [topk]
    int s2;                // valid key rows of the batch
    int topk;
    int64_t kbase;         // key-map row of the batch's key 0 for this key head
    int n2;
};

__device__ __forceinline__ LiUnit li_unit(const LiArgs &A, int t, int n2, int b) {
    LiUnit u;
    const int64_t off = ((int64_t)t * A.g.n2 + n2) * A.g.block_count;
    u.idx = A.idx + off;
    u.dy = A.dy + off;
    u.s2 = A.ws.kv_blocks[b];
    u.topk = A.g.block_count;
    u.kbase = (int64_t)A.ws.cu_kv[b] * A.g.n2 + n2;
    u.n2 = A.g.n2;
    return u;
}

// Id of selection j (-1 past topk).
__device__ __forceinline__ int li_id(const LiUnit &u, int j) { return j < u.topk ? __ldg(u.idx + j) : -1; }

// Key row (of the [T2 * n2] rows of the key map) of a selection id, or -1 for
// an empty slot or an id out of range (reported when `report`).
__device__ __forceinline__ int64_t li_row(const LiArgs &A, const LiUnit &u, int id, bool report) {
    if (id == -1) return -1;
    if (id < 0 || id >= u.s2) {
        if (report) raise_error(&A.ws.hdr->error, SAG_ERR_INDEX);
        return -1;
    }
    return u.kbase + (int64_t)id * u.n2;
}

template <bool kFp16>
__global__ void __launch_bounds__(kLiThreads, 1)
    k_lig_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k, LiArgs A) {
    using L = LiSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_BAR + 8 * L_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_BAR + 8 * L_COUNT + 4);
    float *wbuf = reinterpret_cast<float *>(smem + L::OFF_W);
    const Geometry &g = A.g;
    const Workspace &ws = A.ws;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = g.group;
    const uint32_t sbase = tc::smem_u32(smem);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < L_COUNT; ++i) {
            const bool two_loaders = i >= L_K_FULL0 && i < L_K_FULL0 + kLiKStages;
            const bool from_threads = i == L_R_FULL0 || i == L_R_FULL1 || i == L_DK_FREE0 || i == L_DK_FREE1 ||
                                      i == L_DQ_FREE0 || i == L_DQ_FREE1;
            tc::mbar_init(&bars[i], from_threads ? 128 : two_loaders ? 2 : 1);
        }
        tc::fence_mbar_init();
    }
    // head rows G..63 of the query stages are never loaded: they stay zero, so
    // the padded heads give S = 0 and R = 0
    if (G < kLiHeads) {
        for (int i = threadIdx.x; i < 2 * L::Q_STAGE / 16; i += kLiThreads)
            reinterpret_cast<uint4 *>(smem + L::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
        tc::fence_proxy_async_smem();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&]() {
        *abort_flag = 1;
        raise_error(&ws.hdr->error, SAG_ERR_TIMEOUT);
    };
    // unit -> (token, key head, batch); padding tokens (BSND) are skipped by every role
    auto unit = [&](int64_t u, int &t, int &n2, int &b) {
        t = (int)(u / g.n2);
        n2 = (int)(u % g.n2);
        b = batch_of(ws.cu_q, g.batch, t);
        return t < ws.q_end[b];
    };

    if (warp == 0 || warp == kLiLoader2) {
        // ------------------------------------------------------ TMA producers
        // Warp 0 loads the query tile and weights of each unit and the first
        // 64 dims of every gathered key row; warp 10 the other 64 dims.  Each
        // arms the key-stage barrier with its own bytes.
        const bool lead = warp == 0;
        const int h = lead ? 0 : 1;
        if (lead && lane == 0) {
            tc::prefetch_tmap(&map_q);
            tc::prefetch_tmap(&map_k);
        }
        int uu = 0, kc = 0;
        uint32_t armed_q[2] = {0, 0}, armed_k[kLiKStages] = {};
        bool ok = true;
        for (int64_t u = blockIdx.x; u < A.n_units && ok; u += gridDim.x) {
            int t, n2, b;
            if (!unit(u, t, n2, b)) continue;
            const LiUnit lu = li_unit(A, t, n2, b);
            const int qs = uu & 1;
            if (lead) {
                if (uu >= 2 && !tc::mbar_wait(&bars[L_Q_EMPTY0 + qs], ((uu >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                // the unit's weights (0 past G) for the relu warps; the arrive below
                // publishes them with the query tile
                for (int hh = lane; hh < kLiHeads; hh += 32)
                    wbuf[qs * kLiHeads + hh] = hh < G ? u16_to_f<kFp16>(A.w[(int64_t)t * g.n1 + n2 * G + hh]) : 0.f;
                __syncwarp();
                ++armed_q[qs];
                if (lane == 0) {
                    tc::mbar_arrive_expect_tx(&bars[L_Q_FULL0 + qs], (uint32_t)G * kLiD * 2);
                    for (int c = 0; c < 2; ++c)
                        tc::tma_load_2d(smem + L::OFF_Q + qs * L::Q_STAGE + c * (L::Q_STAGE / 2), &map_q, c * 64,
                                        t * g.n1 + n2 * G, &bars[L_Q_FULL0 + qs]);
                }
            }
            for (int c = 0; c < A.nchunks; ++c, ++kc) {
                const int ks = kc % kLiKStages;
                // the chunk's key rows, read before waiting for the stage; an
                // empty or bad slot fetches the batch's first key row (its R is 0)
                int y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int64_t r = li_row(A, lu, li_id(lu, c * kLiChunk + 4 * lane + e), false);
                    y[e] = (int)(r >= 0 ? r : lu.kbase);
                }
                if (kc >= kLiKStages &&
                    !tc::mbar_wait(&bars[L_K_EMPTY0 + ks], ((kc / kLiKStages) - 1) & 1, abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                ++armed_k[ks];
                if (lane == 0) tc::mbar_arrive_expect_tx(&bars[L_K_FULL0 + ks], (uint32_t)kLiChunk * 64 * 2);
                __syncwarp();
                uint8_t *kdst = smem + L::OFF_K + ks * L::K_STAGE;
                tc::tma_gather4(kdst + h * (L::K_STAGE / 2) + lane * 512, &map_k, h * 64, y[0], y[1], y[2], y[3],
                                &bars[L_K_FULL0 + ks]);
            }
            ++uu;
        }
        if (!ok && lane == 0) fail();
        bool drained = true;
        for (int i = 0; i < 2; ++i) drained = tc::drain_armed(&bars[L_Q_FULL0 + i], armed_q[i], kWaitNs) && drained;
        for (int i = 0; i < kLiKStages; ++i)
            drained = tc::drain_armed(&bars[L_K_FULL0 + i], armed_k[i], kWaitNs) && drained;
        if (!drained) fail();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule; one elected lane issues each
        // tcgen05 instruction (descriptors stay warp-uniform).
        const bool bf16 = !kFp16;
        const uint32_t id_s = tc::idesc_f16(kLiChunk, kLiHeads, bf16, false, false);   // S^T = Kc Q^T
        const uint32_t id_q = tc::idesc_f16(kLiD, kLiHeads, bf16, true, true);         // dQ^T += Kc^T R
        const uint32_t id_k = tc::idesc_f16(kLiChunk, kLiD, bf16, false, true);        // dKc = R Q
        const uint64_t d_k0 = tc::sw128_desc(sbase + L::OFF_K, 16, 1024);                  // key tile, K-major
        const uint64_t d_kt0 = tc::sw128_desc(sbase + L::OFF_K, L::K_STAGE / 2, 1024);     // key tile, MN-major
        const uint64_t d_q0 = tc::sw128_desc(sbase + L::OFF_Q, 16, 1024);                  // query tile, K-major
        const uint64_t d_qt0 = tc::sw128_desc(sbase + L::OFF_Q, L::Q_STAGE / 2, 1024);     // query tile, MN-major
        const uint64_t d_rt0 = tc::sw128_desc(sbase + L::OFF_R, L::R_STAGE, 1024);         // R, MN-major
        const uint64_t d_r0 = tc::sw128_desc(sbase + L::OFF_R, 16, 1024);                  // R, K-major
        auto wait = [&](int bi, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, tc::mbar_wait(&bars[bi], parity, abort_flag, kWaitNs));
        };
        struct Prev { int kc, qs, dqb, uu; bool first, last; };
        Prev pv{};
        bool have = false, ok = true;
        int uu = 0, kc = 0;
        // the dQ / dK MMAs of chunk p once its R is in shared memory
        auto back = [&](const Prev &p) -> bool {
            const int rs = p.kc & 1, ks = p.kc % kLiKStages;
            if (!wait(L_R_FULL0 + rs, (p.kc >> 1) & 1)) return false;
            if (p.first && p.uu >= 2 && !wait(L_DQ_FREE0 + p.dqb, ((p.uu >> 1) - 1) & 1)) return false;
            if (p.kc >= 2 && !wait(L_DK_FREE0 + rs, ((p.kc >> 1) - 1) & 1)) return false;
            tc::tc_fence_after();
            const uint64_t kt = d_kt0 + (uint64_t)((ks * L::K_STAGE) >> 4);
            const uint64_t qt = d_qt0 + (uint64_t)((p.qs * L::Q_STAGE) >> 4);
            const uint64_t rt = d_rt0 + (uint64_t)((rs * L::R_STAGE) >> 4);
            const uint64_t rk = d_r0 + (uint64_t)((rs * L::R_STAGE) >> 4);
            // dQ^T += Kc^T R: A = key tile MN-major (dims x keys), B = R MN-major (heads x keys)
#pragma unroll
            for (int kk = 0; kk < kLiChunk / 16; ++kk)
                tc::mma_f16_ss_warp(tmem + kLiColDQ + p.dqb * kLiHeads, kt + ((kk * 2048) >> 4),
                                    rt + ((kk * 2048) >> 4), id_q, (!p.first) || (kk > 0));
            // dKc = R Q: A = R K-major (keys x heads), B = query tile MN-major (dims x heads)
#pragma unroll
            for (int kk = 0; kk < kLiHeads / 16; ++kk)
                tc::mma_f16_ss_warp(tmem + kLiColDK + rs * kLiD, rk + ((kk * 32) >> 4), qt + ((kk * 2048) >> 4),
                                    id_k, kk > 0);
            tc::mma_commit_warp(&bars[L_DK_FULL0 + rs]);
            tc::mma_commit_warp(&bars[L_K_EMPTY0 + ks]);      // key tile and R stage free
            if (p.last) {
                tc::mma_commit_warp(&bars[L_DQ_FULL0 + p.dqb]);
                tc::mma_commit_warp(&bars[L_Q_EMPTY0 + p.qs]);
            }
            return true;
        };
        for (int64_t u = blockIdx.x; u < A.n_units && ok; u += gridDim.x) {
            int t, n2, b;
            if (!unit(u, t, n2, b)) continue;
            const int qs = uu & 1;
            if (!wait(L_Q_FULL0 + qs, (uu >> 1) & 1)) { ok = false; break; }
            const uint64_t dq = d_q0 + (uint64_t)((qs * L::Q_STAGE) >> 4);
            for (int c = 0; c < A.nchunks; ++c, ++kc) {
                const int ks = kc % kLiKStages;
                if (!wait(L_K_FULL0 + ks, (kc / kLiKStages) & 1)) { ok = false; break; }
                tc::tc_fence_after();
                const uint64_t dk = d_k0 + (uint64_t)((ks * L::K_STAGE) >> 4);
                // S^T = Kc Q^T (both operands K-major)
#pragma unroll
                for (int kk = 0; kk < kLiD / 16; ++kk)
                    tc::mma_f16_ss_warp(tmem + kLiColS + (kc & 1) * kLiHeads,
                                        dk + ((((kk >> 2) * (L::K_STAGE / 2)) + (kk & 3) * 32) >> 4),
                                        dq + ((((kk >> 2) * (L::Q_STAGE / 2)) + (kk & 3) * 32) >> 4), id_s, kk > 0);
                tc::mma_commit_warp(&bars[L_S_FULL0 + (kc & 1)]);
                if (have && !back(pv)) { ok = false; break; }
                pv = Prev{kc, qs, uu & 1, uu, c == 0, c == A.nchunks - 1};
                have = true;
            }
            ++uu;
        }
        if (ok && have && !back(pv)) ok = false;
        if (!ok && lane == 0) fail();
        tc::mma_commit_warp(&bars[L_DRAIN]);
        if (!__all_sync(0xffffffffu, tc::mbar_wait_drain(&bars[L_DRAIN], 0, kWaitNs)) && lane == 0) fail();
    } else if (warp < 6) {
        // ------------------------------------------------------ relu / dW
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                        // key of the chunk = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        int uu = 0, kc = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < A.n_units && ok; u += gridDim.x) {
            int t, n2, b;
            if (!unit(u, t, n2, b)) continue;
            // the weights come with the query tile (stage = unit parity)
            ok = tc::mbar_wait(&bars[L_Q_FULL0 + (uu & 1)], (uu >> 1) & 1, abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const float *wv = wbuf + (uu & 1) * kLiHeads;
            const LiUnit lu = li_unit(A, t, n2, b);
            float dw0 = 0.f, dw1 = 0.f;                      // this lane's two heads (see below)
            // this key's id and dy, one chunk ahead of the chunk being processed
            int id_next = li_id(lu, r);
            float dy_next = r < lu.topk ? __ldg(lu.dy + r) : 0.f;
            for (int c = 0; c < A.nchunks; ++c, ++kc) {
                const int ks = kc & 1;
                const int id = id_next;
                const float dy_c = dy_next;
                if (c + 1 < A.nchunks) {
                    const int j = (c + 1) * kLiChunk + r;
                    id_next = li_id(lu, j);
                    dy_next = j < lu.topk ? __ldg(lu.dy + j) : 0.f;
                }
                const float dyv = li_row(A, lu, id, true) >= 0 ? dy_c : 0.f;
                ok = tc::mbar_wait(&bars[L_S_FULL0 + ks], (kc >> 1) & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                float v[kLiHeads];                           // relu(S) * dy, reduced below
                uint32_t pk[kLiHeads / 2];
#pragma unroll
                for (int h0 = 0; h0 < kLiHeads; h0 += 32) {
                    uint32_t sv[4][8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) tc::tmem_ld8(trow + kLiColS + ks * kLiHeads + h0 + 8 * i, sv[i]);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const int h = h0 + 8 * i + e;
                            const float x0 = __uint_as_float(sv[i][e]), x1 = __uint_as_float(sv[i][e + 1]);
                            v[h] = fmaxf(x0, 0.f) * dyv;
                            v[h + 1] = fmaxf(x1, 0.f) * dyv;
                            const float r0 = x0 > 0.f ? dyv * wv[h] : 0.f;
                            const float r1 = x1 > 0.f ? dyv * wv[h + 1] : 0.f;
                            pk[h / 2] = pack2<kFp16>(r0, r1);
                        }
                }
                // R row of this key into the chunk's R stage (128-byte swizzled rows)
                uint8_t *rrow = smem + L::OFF_R + ks * L::R_STAGE;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4 *>(rrow + sw_off(r, cc)) =
                        make_uint4(pk[cc * 4], pk[cc * 4 + 1], pk[cc * 4 + 2], pk[cc * 4 + 3]);
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[L_R_FULL0 + ks]);
                // dW over the warp's 32 keys: each step trades half of the
                // values with the partner lane (the upper half of the heads goes
                // to the lane with the step's bit set) and adds; after 5 steps
                // lane l holds heads 2 l and 2 l + 1 summed over all 32 lanes
#pragma unroll
                for (int step = 0; step < 5; ++step) {
                    const int off = 16 >> step, half = 32 >> step;
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const float send = upper ? v[i] : v[i + half];
                        const float keep = upper ? v[i + half] : v[i];
                        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
                dw0 += v[0];
                dw1 += v[1];
            }
            if (!ok) break;
            // lane l holds heads 2 l and 2 l + 1 summed over its warp's keys
            float *dwa = ws.dkv_acc + (int64_t)t * g.n1 + n2 * G;
            if (2 * lane < G) atomicAdd(dwa + 2 * lane, dw0);
            if (2 * lane + 1 < G) atomicAdd(dwa + 2 * lane + 1, dw1);
            ++uu;
        }
        if (!ok) fail();
    } else {
        // ------------------------------------------------------ epilogue
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                        // key of the chunk / head dim = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        uint8_t *stg = smem + L::OFF_STG + (warp - 6) * 4096;
        float *acc = ws.dq_acc;                              // fp32 dK [T2 * n2, d]
        int uu = 0, kc = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < A.n_units && ok; u += gridDim.x) {
            int t, n2, b;
            if (!unit(u, t, n2, b)) continue;
            const LiUnit lu = li_unit(A, t, n2, b);
            for (int c = 0; c < A.nchunks; ++c, ++kc) {
                const int ks = kc & 1;
                const int64_t krow = li_row(A, lu, li_id(lu, c * kLiChunk + r), false);
                ok = tc::mbar_wait(&bars[L_DK_FULL0 + ks], (kc >> 1) & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                for (int c32 = 0; c32 < kLiD / 32; ++c32) {
                    uint32_t v0[16], v1[16];
                    tc::tmem_ld16(trow + kLiColDK + ks * kLiD + c32 * 32, v0);
                    tc::tmem_ld16(trow + kLiColDK + ks * kLiD + c32 * 32 + 16, v1);
                    tc::tmem_wait_ld();
                    // stage the warp's 32 keys x 32 dims, then reduce whole 128-byte row segments
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4)
                        *reinterpret_cast<uint4 *>(stg + lane * 128 + ((j4 ^ (lane & 7)) << 4)) =
                            make_uint4(v0[4 * j4], v0[4 * j4 + 1], v0[4 * j4 + 2], v0[4 * j4 + 3]);
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4)
                        *reinterpret_cast<uint4 *>(stg + lane * 128 + (((j4 + 4) ^ (lane & 7)) << 4)) =
                            make_uint4(v1[4 * j4], v1[4 * j4 + 1], v1[4 * j4 + 2], v1[4 * j4 + 3]);
                    __syncwarp();
#pragma unroll
                    for (int kq = 0; kq < 8; ++kq) {
                        const int rr = kq * 4 + (lane >> 3), j4 = lane & 7;
                        const int64_t kr = __shfl_sync(0xffffffffu, krow, rr);
                        const float4 x = *reinterpret_cast<const float4 *>(stg + rr * 128 + ((j4 ^ (rr & 7)) << 4));
                        if (kr >= 0) tc::red_add_v4(acc + kr * kLiD + c32 * 32 + j4 * 4, x.x, x.y, x.z, x.w);
                    }
                    __syncwarp();
                }
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[L_DK_FREE0 + ks]);
            }
            if (!ok) break;
            // dQ of the unit: lane = head dim, columns = heads
            const int dqb = uu & 1;
            ok = tc::mbar_wait(&bars[L_DQ_FULL0 + dqb], (uu >> 1) & 1, abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc::tc_fence_after();
            for (int h0 = 0; h0 < kLiHeads; h0 += 16) {
                if (h0 >= G) break;
                uint32_t v[16];
                tc::tmem_ld16(trow + kLiColDQ + dqb * kLiHeads + h0, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (h0 + i < G)
                        A.dq[((int64_t)t * g.n1 + n2 * G + h0 + i) * kLiD + r] = f_to_u16<kFp16>(__uint_as_float(v[i]));
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&bars[L_DQ_FREE0 + dqb]);
            ++uu;
        }
        if (!ok) fail();
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// fp32 dK accumulator -> 16-bit dk
template <bool kFp16>
__global__ void __launch_bounds__(256) k_lig_cast(const float *__restrict__ in, uint16_t *__restrict__ out, int64_t n4) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = reinterpret_cast<const float4 *>(in)[i];
        ushort4 o;
        o.x = f_to_u16<kFp16>(v.x);
        o.y = f_to_u16<kFp16>(v.y);
        o.z = f_to_u16<kFp16>(v.z);
        o.w = f_to_u16<kFp16>(v.w);
        reinterpret_cast<ushort4 *>(out)[i] = o;
    }
}

template <bool kFp16>
__global__ void __launch_bounds__(256) k_lig_cast1(const float *__restrict__ in, uint16_t *__restrict__ out, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = f_to_u16<kFp16>(in[i]);
}

template <bool kFp16>
cudaError_t launch_lig_t(const Geometry &g, const Workspace &ws, const sli_io &io, cudaStream_t s, int num_sms) {
    LiArgs a;
    a.g = g;
    a.ws = ws;
    a.idx = io.indices;
    a.dy = io.dy;
    a.w = (const uint16_t *)io.weights;
    a.dq = (uint16_t *)io.dq;
    a.n_units = (int64_t)g.t1 * g.n2;
    a.nchunks = (g.block_count + kLiChunk - 1) / kLiChunk;
    CUtensorMap mq, mk;
    if (!tmap_2d(&mq, io.query, kFp16, kLiD, (uint64_t)g.t1 * g.n1, g.group) ||
        !tmap_2d(&mk, io.key, kFp16, kLiD, (uint64_t)g.t2 * g.n2, 1))
        return cudaErrorInvalidValue;
    auto fn = k_lig_tc<kFp16>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, LiSmem::TOTAL);
    if (e != cudaSuccess) return e;
    int64_t grid = a.n_units < num_sms ? a.n_units : num_sms;
    if (grid < 1) grid = 1;
    fn<<<(int)grid, kLiThreads, LiSmem::TOTAL, s>>>(mq, mk, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto cast = [&](const float *in, void *out, int64_t n) {
        const int64_t n4 = n / 4;
        int64_t cg = (n4 + 255) / 256;
        if (cg > (int64_t)num_sms * 8) cg = (int64_t)num_sms * 8;
        if (cg > 0) k_lig_cast<kFp16><<<(int)cg, 256, 0, s>>>(in, (uint16_t *)out, n4);
    };
    cast(ws.dq_acc, io.dk, (int64_t)g.t2 * g.n2 * kLiD);
    const int64_t nw = (int64_t)g.t1 * g.n1;
    int64_t cw = (nw + 255) / 256;
    if (cw > (int64_t)num_sms * 8) cw = (int64_t)num_sms * 8;
    if (cw > 0) k_lig_cast1<kFp16><<<(int)cw, 256, 0, s>>>(ws.dkv_acc, (uint16_t *)io.dweights, nw);
    return cudaGetLastError();
}

}  // namespace

bool lig_tc_supported(const Geometry &g) { return g.d_qk == kLiD && g.group >= 1 && g.group <= kLiHeads; }

cudaError_t launch_lig(const Geometry &g, const Workspace &ws, const sli_io &io, bool fp16, cudaStream_t s,
                       int num_sms) {
    if (!lig_tc_supported(g)) return cudaErrorInvalidValue;
    return fp16 ? launch_lig_t<true>(g, ws, io, s, num_sms) : launch_lig_t<false>(g, ws, io, s, num_sms);
}

}  // namespace sag
