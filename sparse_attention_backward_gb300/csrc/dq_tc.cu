// Deterministic dQ on the tensor cores, from the dS the main kernel stored.
//
// dQ[t, n2*G + g] = scale * sum_slot sum_r dS[t][n2][slot][g][r] * K[row(slot, r), n2]
// ("NsaSelectedAttentionGrad" README, function description: dQ = dS K / sqrt(d)
// over the gathered rows).  One (token, KV head) pair at a time:
//     dQ^T [Dqk x G] += K_slot^T [Dqk x bs] . dS_slot^T [bs x G]
// as tcgen05.mma with M = Dqk rows (128, or 128 + the [64,192) half for 192),
// N = G rounded up to 16 (columns past G are never read), K = bs keys; slots
// and keys are accumulated in one fixed order, so the result is the same
// bits on every run.  A persistent CTA: warp 0 loads each slot's key block and
// dS tile with TMA into a 3-stage ring, warp 1 issues the MMAs into one of
// two TMEM accumulators, warps 2-5 read the finished accumulator and write dQ.
#include "kernels.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace sag {
namespace {

constexpr int kDqThreads = 192;
constexpr int kStages = 3;
constexpr uint64_t kDqWaitNs = 2000000000ull;

// A stage holds 64 keys of one selected block (a 128-key block takes two
// stages): the key rows, KC chunks of 64 rows x 128 B, and the dS plane of
// those keys, up to 32 rows x 128 B.
constexpr int kSub = 64;

template <int DQK>
struct DqSmem {
    static constexpr int KC = DQK / 64;
    static constexpr int K_BYTES = KC * kSub * 128;
    static constexpr int DS_BYTES = 32 * 128;
    static constexpr int STAGE = K_BYTES + DS_BYTES;
    static constexpr int OFF_BAR = kStages * STAGE;
    static constexpr int TOTAL = OFF_BAR + 256 + 1024;
    // two CTAs per SM (their shared memory fits): two MMA warps then issue
    // the pass's small MMAs side by side
    static constexpr int CTAS_PER_SM = 2 * (TOTAL + 1024) <= 227 * 1024 ? 2 : 1;
};

enum DqBar { D_FULL0 = 0, D_EMPTY0 = kStages, D_ACC_FULL0 = 2 * kStages, D_ACC_FREE0 = 2 * kStages + 2,
             D_DRAIN = 2 * kStages + 4, D_COUNT = 2 * kStages + 5 };

struct DqArgs {
    Geometry g;
    Workspace ws;
    const int32_t *topk;
    uint16_t *dq, *dq_rope;
    int n_pad;          // G rounded up to a multiple of 16
};

__device__ __forceinline__ bool slot_ok(const Geometry &g, const Workspace &ws, const int32_t *topk,
                                        int64_t pair, int slot, int nblk) {
    const int id = __ldg(topk + pair * g.block_count + slot);
    return id >= 0 && id < nblk;
}

template <bool kFp16, int DQK, int BS>
__global__ void __launch_bounds__(kDqThreads, DqSmem<DQK>::CTAS_PER_SM)
    k_dq_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_ds,
            const __grid_constant__ CUtensorMap map_kr, DqArgs A) {
    using L = DqSmem<DQK>;
    constexpr int KC = L::KC;
    constexpr int kSubs = BS / kSub;   // stages per selected block
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_BAR + 8 * D_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_BAR + 8 * D_COUNT + 4);
    const Geometry &g = A.g;
    const Workspace &ws = A.ws;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = g.group;
    const int64_t npairs = (int64_t)(g.tok_hi - g.tok_lo) * g.n2;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&bars[D_FULL0 + s], 1);
            tc::mbar_init(&bars[D_EMPTY0 + s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&bars[D_ACC_FULL0 + b], 1);
            tc::mbar_init(&bars[D_ACC_FREE0 + b], 128);
        }
        tc::mbar_init(&bars[D_DRAIN], 1);
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 128);
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
    // accumulator b: dims [0,128) at column 64*b, dims [64,192) at 64*b + 32
    auto acc_col = [&](int b, int hi) { return (uint32_t)(64 * b + 32 * hi); };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::prefetch_tmap(&map_k);
            tc::prefetch_tmap(&map_ds);
            if (g.d_rope) tc::prefetch_tmap(&map_kr);
            int it = 0;
            uint32_t armed[kStages] = {};
            bool ok = true;
            for (int64_t cp = blockIdx.x; cp < npairs && ok; cp += gridDim.x) {
                const int t = g.tok_lo + (int)(cp / g.n2), n2 = (int)(cp % g.n2);
                const int64_t pair = (int64_t)t * g.n2 + n2;
                const int b = batch_of(ws.cu_q, g.batch, t);
                const int nblk = t < ws.q_end[b] ? ws.kv_blocks[b] : 0;   // ids must be below; none for padding
                for (int slot = 0; slot < g.block_count && ok; ++slot) {
                    if (!slot_ok(g, ws, A.topk, pair, slot, nblk)) continue;
                    const int id = __ldg(A.topk + pair * g.block_count + slot);
                    const int dsrow = (int)(((int64_t)cp * g.block_count + slot) * G);
                    for (int h = 0; h < kSubs; ++h) {
                        const int s = it % kStages;
                        if (it >= kStages &&
                            !tc::mbar_wait(&bars[D_EMPTY0 + s], ((it / kStages) - 1) & 1, abort_flag, kDqWaitNs)) {
                            ok = false;
                            break;
                        }
                        const int key0 = ws.cu_kv[b] + id * BS + h * kSub;
                        uint8_t *st = smem + s * L::STAGE;
                        ++armed[s];
                        tc::mbar_arrive_expect_tx(&bars[D_FULL0 + s], (uint32_t)(kSub * DQK * 2 + G * kSub * 2));
                        for (int c = 0; c < KC; ++c)
                            tc::tma_load_3d(st + c * kSub * 128, (g.d_rope && c == 2) ? &map_kr : &map_k,
                                            (g.d_rope && c == 2) ? 0 : c * 64, n2, key0, &bars[D_FULL0 + s]);
                        tc::tma_load_2d(st + L::K_BYTES, &map_ds, h * kSub, dsrow, &bars[D_FULL0 + s]);
                        ++it;
                    }
                }
            }
            if (!ok) fail();
            // let every load issued land before the CTA exits
            bool drained = true;
            for (int i = 0; i < kStages; ++i) drained = tc::drain_armed(&bars[D_FULL0 + i], armed[i], kDqWaitNs) && drained;
            if (!drained) fail();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule; one elected lane issues each
        // instruction (a pair is 8-16 small MMAs per slot: the issue rate
        // matters).
        const uint32_t idesc = tc::idesc_f16(128, A.n_pad, !kFp16, true, false);
        auto wait = [&](int b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, tc::mbar_wait(&bars[b], parity, abort_flag, kDqWaitNs));
        };
        int it = 0, np = 0;
        bool ok = true;
        for (int64_t cp = blockIdx.x; cp < npairs && ok; cp += gridDim.x, ++np) {
            const int t = g.tok_lo + (int)(cp / g.n2), n2 = (int)(cp % g.n2);
            const int64_t pair = (int64_t)t * g.n2 + n2;
            const int b = batch_of(ws.cu_q, g.batch, t);
            const int nblk = t < ws.q_end[b] ? ws.kv_blocks[b] : 0;   // ids must be below; none for padding
            const int ab = np & 1;
            if (np >= 2 && !wait(D_ACC_FREE0 + ab, ((np >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            bool first = true;
            for (int slot = 0; slot < g.block_count && ok; ++slot) {
                if (!slot_ok(g, ws, A.topk, pair, slot, nblk)) continue;
                for (int h = 0; h < kSubs; ++h) {
                    const int s = it % kStages;
                    if (!wait(D_FULL0 + s, (it / kStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t kst = tc::smem_u32(smem + s * L::STAGE);
                    const uint32_t dst = kst + L::K_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kSub / 16; ++kk) {
                        // A = K^T (dims x keys, MN-major), B = dS^T (keys x G, K-major)
                        const uint64_t bdesc = tc::sw128_desc(dst + kk * 32, 16, 1024);
                        tc::mma_f16_ss_warp(tmem + acc_col(ab, 0), tc::sw128_desc(kst + kk * 2048, kSub * 128, 1024),
                                            bdesc, idesc, !first || kk > 0);
                        if (DQK == 192)
                            tc::mma_f16_ss_warp(tmem + acc_col(ab, 1),
                                                tc::sw128_desc(kst + kSub * 128 + kk * 2048, kSub * 128, 1024), bdesc,
                                                idesc, !first || kk > 0);
                    }
                    tc::mma_commit_warp(&bars[D_EMPTY0 + s]);
                    first = false;
                    ++it;
                }
            }
            if (!ok) break;
            tc::mma_commit_warp(&bars[D_ACC_FULL0 + ab]);
        }
        if (!ok && lane == 0) fail();
        // every MMA issued must be complete before TMEM is freed
        tc::mma_commit_warp(&bars[D_DRAIN]);
        if (!__all_sync(0xffffffffu, tc::mbar_wait_drain(&bars[D_DRAIN], 0, kDqWaitNs)) && lane == 0) fail();
    } else {
        // ------------------------------------------------------ epilogue
        const int q4 = warp & 3;
        const int d = q4 * 32 + lane;                  // TMEM lane = head dim
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        int np = 0;
        bool ok = true;
        for (int64_t cp = blockIdx.x; cp < npairs && ok; cp += gridDim.x, ++np) {
            const int t = g.tok_lo + (int)(cp / g.n2), n2 = (int)(cp % g.n2);
            const int64_t pair = (int64_t)t * g.n2 + n2;
            const int b = batch_of(ws.cu_q, g.batch, t);
            const int nblk = t < ws.q_end[b] ? ws.kv_blocks[b] : 0;   // ids must be below; none for padding
            int nvalid = 0;
            for (int slot = 0; slot < g.block_count; ++slot) nvalid += slot_ok(g, ws, A.topk, pair, slot, nblk);
            const int ab = np & 1;
            const bool w = tc::mbar_wait(&bars[D_ACC_FULL0 + ab], (np >> 1) & 1, abort_flag, kDqWaitNs);
            ok = __all_sync(0xffffffffu, w);
            if (!ok) break;
            tc::tc_fence_after();
            const int64_t row0 = (int64_t)t * g.n1 + (int64_t)n2 * G;   // first dq row of the pair
            for (int g0 = 0; g0 < G; g0 += 16) {
                uint32_t lo[16], hi[16];
                tc::tmem_ld16(trow + acc_col(ab, 0) + g0, lo);
                if (DQK == 192) tc::tmem_ld16(trow + acc_col(ab, 1) + g0, hi);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (g0 + j >= G) break;
                    const float vlo = nvalid ? __uint_as_float(lo[j]) : 0.f;
                    *split_col(A.dq, A.dq_rope, row0 + g0 + j, d, DQK, g.d_rope) = f_to_u16<kFp16>(vlo * g.scale);
                    if (DQK == 192 && d >= 64) {
                        const float vhi = nvalid ? __uint_as_float(hi[j]) : 0.f;
                        *split_col(A.dq, A.dq_rope, row0 + g0 + j, 64 + d, DQK, g.d_rope) =
                            f_to_u16<kFp16>(vhi * g.scale);
                    }
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&bars[D_ACC_FREE0 + ab]);
        }
        if (!ok) fail();
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 128);
    }
}

template <bool kFp16, int DQK, int BS>
static cudaError_t launch_dq_tc_t(const Geometry &g, const Workspace &ws, const sag_io &io, cudaStream_t s,
                                  int num_sms) {
    const int64_t npairs = (int64_t)(g.tok_hi - g.tok_lo) * g.n2;
    if (npairs == 0) return cudaSuccess;
    DqArgs a;
    a.g = g;
    a.ws = ws;
    a.topk = io.topk_indices;
    a.dq = (uint16_t *)io.dq;
    a.dq_rope = (uint16_t *)io.dq_rope;
    a.n_pad = (g.group + 15) / 16 * 16;
    CUtensorMap mk, mkr, mds;
    const uint64_t ds_rows = (uint64_t)npairs * g.block_count * g.group;
    const uint64_t d_main = (uint64_t)(g.d_qk - g.d_rope);
    if (!tmap_3d(&mk, io.key, kFp16, d_main, g.n2, g.t2, kSub) || !tmap_2d(&mds, ws.ds, kFp16, BS, ds_rows, g.group))
        return cudaErrorInvalidValue;
    if (g.d_rope) {
        if (!tmap_3d(&mkr, io.key_rope, kFp16, g.d_rope, g.n2, g.t2, kSub)) return cudaErrorInvalidValue;
    } else {
        mkr = mk;
    }
    auto fn = k_dq_tc<kFp16, DQK, BS>;
    const int smem = DqSmem<DQK>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)num_sms * DqSmem<DQK>::CTAS_PER_SM;
    const int64_t grid = npairs < slots ? npairs : slots;
    fn<<<(int)grid, kDqThreads, smem, s>>>(mk, mds, mkr, a);
    return cudaGetLastError();
}

}  // namespace

bool dq_tc_supported(const Geometry &g) {
    return (g.d_qk == 128 || g.d_qk == 192) && (g.block_size == 64 || g.block_size == 128) && g.group <= 32;
}

cudaError_t launch_dq_tc(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, cudaStream_t s,
                         int num_sms) {
#define SAG_DQ_CASE(F, D, B) \
    if (fp16 == F && g.d_qk == D && g.block_size == B) return launch_dq_tc_t<F, D, B>(g, ws, io, s, num_sms);
    SAG_DQ_CASE(false, 192, 64) SAG_DQ_CASE(false, 192, 128) SAG_DQ_CASE(false, 128, 64)
    SAG_DQ_CASE(false, 128, 128) SAG_DQ_CASE(true, 192, 64) SAG_DQ_CASE(true, 192, 128)
    SAG_DQ_CASE(true, 128, 64) SAG_DQ_CASE(true, 128, 128)
#undef SAG_DQ_CASE
    return cudaErrorInvalidValue;
}

}  // namespace sag
