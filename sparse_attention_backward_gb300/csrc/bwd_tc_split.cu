// Tensor-core key-block-major backward with the softmax split in two phases
// (the schedule taken for small query groups; bwd_tc.cu has the other one).
//
// Same work units, data layout, warp roles and MMAs as bwd_tc.cu (that file's
// header lists the per-tile products and their sources).  The difference is
// the order: the MMA warp issues, per query tile t,
//     S(t) | dK, dQ (t-1) | dP(t) | dV(t)
// and the softmax works in two phases, P = exp2(S * scale*log2e - lse2) as
// soon as S(t) is in TMEM (S's columns are released once read, so S(t+1) can
// follow), then dS = P (dP - Delta) once dP(t) is in.  The softmax thus runs
// beside the tensor pipe instead of between its groups; the price is that the
// Q tile of t+1 can only be fetched once dK(t-1) has retired, which exposes
// load latency when Q rows come from DRAM in 2 KB boxes (large groups) and
// pays off when the rows are gathered four at a time (G <= 4).  Q and dY are
// signalled per 64-column chunk, and the MMA warp runs convergent with one
// elected lane issuing each tcgen05 instruction.
#include <stdlib.h>

#include <type_traits>

#include "kernels.cuh"
#include "tc.cuh"
#include "tile.cuh"
#include "tmap.cuh"

namespace sag {
namespace {

constexpr int kMeta = 4;            // depth of the tile-metadata ring
// Warps: 0 lead producer, 1 MMA, 2-5 softmax, 6-9 epilogue, 10-11 loaders
// (12 warps: three per SM sub-partition, so 168 registers a thread fit)
constexpr int kLoaders = 3;
constexpr int kLoaderWarp1 = 10;
constexpr int kSplitThreads = (kLoaderWarp1 + kLoaders - 1) * 32;

// TMEM columns (512 allocated)
constexpr uint32_t kColS = 0, kColDP = 64, kColDV = 128, kColDKlo = 192, kColDKhi = 256, kColDQ = 320;

template <int DQK>
struct Smem {
    static constexpr int KC = DQK / 64;                  // 64-wide chunks of a q / k row
    static constexpr int DOS = (DQK == 128) ? 2 : 1;     // dY stages
    static constexpr int K_TILE = KC * 8192;             // 64 rows x 128 B per chunk
    static constexpr int V_TILE = 2 * 8192;
    static constexpr int Q_STAGE = KC * 16384;           // 128 rows x 128 B per chunk
    static constexpr int DO_STAGE = 2 * 16384;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + K_TILE;
    static constexpr int OFF_Q = OFF_V + V_TILE;
    static constexpr int OFF_DO = OFF_Q + 2 * Q_STAGE;
    static constexpr int OFF_P = OFF_DO + DOS * DO_STAGE;
    static constexpr int OFF_DS = OFF_P + 16384;
    static constexpr int OFF_STG = OFF_DS + 16384;       // 4 epilogue warps x 4 KB
    static constexpr int OFF_META = OFF_STG + 16384;     // kMeta x 128 ints
    static constexpr int OFF_RING = OFF_META + kMeta * kRows * 4;   // kURing unit ids
    static constexpr int OFF_LENT = OFF_RING + 64;                   // kLoaders x 128 ints
    static constexpr int OFF_BAR = OFF_LENT + kLoaders * kRows * 4;
    static constexpr int TOTAL = OFF_BAR + 512 + 1024;   // + slack for 1024-B alignment
};

// S_FREE: the softmax has read S (TMEM columns reusable); P_FULL / DS_FULL:
// P / dS are in shared memory; P_FREE / DS_FREE: the MMAs reading them are
// done; DP_FULL: dP is in TMEM; MMA_DONE: dQ is in TMEM; DQ_FREE: drained.
// Q_FULL / DO_FULL are per stage and 64-column chunk (stage * 3 + chunk,
// stage * 2 + chunk), so the MMAs start on the first chunk of a tile.
enum Bar {
    B_KV_FULL = 0, B_KV_EMPTY, B_Q_FULL, B_Q_EMPTY0 = B_Q_FULL + 6, B_Q_EMPTY1, B_DO_FULL,
    B_DO_EMPTY0 = B_DO_FULL + 4, B_DO_EMPTY1, B_S_FULL, B_S_FREE, B_P_FULL, B_P_FREE, B_DP_FULL, B_DS_FULL,
    B_DS_FREE, B_MMA_DONE, B_DQ_FREE, B_ACC_FULL, B_ACC_FREE, B_DRAIN, B_U_FULL, B_U_EMPTY = B_U_FULL + kURing,
    B_COUNT = B_U_EMPTY + kURing
};
// warps that read the unit ring: MMA, 4 softmax, 4 epilogue, the other loaders
constexpr int kRingReaders = 9 + kLoaders - 1;

struct TcArgs {
    Geometry g;
    Workspace ws;
    uint16_t *dk, *dv, *dk_rope;
    int nk, halves, tpt, deterministic;
    int64_t n_titems;
};

template <bool kFp16, int DQK>
__global__ void __launch_bounds__(kSplitThreads, 1)
    k_bwd_tc_split(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
             const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
             const __grid_constant__ CUtensorMap map_qr, const __grid_constant__ CUtensorMap map_kr, TcArgs A) {
    using L = Smem<DQK>;
    constexpr int DV = 128;
    constexpr int KC = L::KC;
    constexpr int DOS = L::DOS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_BAR + 8 * B_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_BAR + 8 * B_COUNT + 4);
    int *meta = reinterpret_cast<int *>(smem + L::OFF_META);
    const Geometry &g = A.g;
    const Workspace &ws = A.ws;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = A.nk, tpt = A.tpt, G = g.group;
    const bool det = A.deterministic != 0;
    // fixed-order dQ: from the stored dS (a later pass re-reads the key
    // blocks), or from per-slot fp32 partials of dQ = dS K stored here
    const bool store_ds = det && !g.dq_slots;
    const uint32_t sbase = tc::smem_u32(smem);
    // 64-column chunk c of a q / k row: the main tensor at column 64 c, or
    // with the rope split chunk 2 from the rope tensor at column 0
    const bool rope = g.d_rope != 0;
    auto qmap = [&](int c) { return (rope && c == 2) ? &map_qr : &map_q; };
    auto kmap = [&](int c) { return (rope && c == 2) ? &map_kr : &map_k; };
    auto cx = [&](int c) { return (rope && c == 2) ? 0 : c * 64; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        tc::mbar_init(&bars[B_KV_FULL], 1);
        tc::mbar_init(&bars[B_KV_EMPTY], 1);
        for (int s = 0; s < 2; ++s) {
            for (int c = 0; c < 3; ++c) tc::mbar_init(&bars[B_Q_FULL + s * 3 + c], kLoaders);
            for (int c = 0; c < 2; ++c) tc::mbar_init(&bars[B_DO_FULL + s * 2 + c], kLoaders);
            tc::mbar_init(&bars[B_Q_EMPTY0 + s], 1);
            tc::mbar_init(&bars[B_DO_EMPTY0 + s], 1);
        }
        tc::mbar_init(&bars[B_S_FULL], 1);
        tc::mbar_init(&bars[B_S_FREE], 128);
        tc::mbar_init(&bars[B_P_FULL], 128);
        tc::mbar_init(&bars[B_P_FREE], 1);
        tc::mbar_init(&bars[B_DP_FULL], 1);
        tc::mbar_init(&bars[B_DS_FULL], 128);
        tc::mbar_init(&bars[B_DS_FREE], 1);
        tc::mbar_init(&bars[B_MMA_DONE], 1);
        tc::mbar_init(&bars[B_DQ_FREE], 128);
        tc::mbar_init(&bars[B_ACC_FULL], 1);
        tc::mbar_init(&bars[B_ACC_FREE], 128);
        tc::mbar_init(&bars[B_DRAIN], 1);
        for (int q = 0; q < kURing; ++q) {
            tc::mbar_init(&bars[B_U_FULL + q], 1);
            tc::mbar_init(&bars[B_U_EMPTY + q], kRingReaders);
        }
        tc::fence_mbar_init();
    }
    // rows of a Q / dY tile no token fills (when G does not divide 128) must
    // hold finite values: zero the staging buffers once
    if (tpt * G < kRows) {
        for (int i = threadIdx.x; i < (2 * L::Q_STAGE + DOS * L::DO_STAGE) / 16; i += kSplitThreads)
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
    // work units come from the launch's ticket counter (hot buckets are much
    // larger than cold ones: a static split would leave SMs idle)
    const UnitRing ring{reinterpret_cast<int64_t *>(smem + L::OFF_RING), &bars[B_U_FULL], &bars[B_U_EMPTY]};

    if (warp == 0 || warp >= kLoaderWarp1) {
        // ------------------------------------------------------ TMA producers
        // kLoaders warps share each tile's query-side loads: one warp issues a
        // gather4 (or a token box) about every 70 cycles, which alone would
        // bound the small-group tiles.  Warp 0 leads: it takes the units from
        // the ticket counter, loads the K / V tile and writes the tile's
        // metadata; every loader arms each Q / dY barrier with its own bytes.
        const int lq = warp == 0 ? 0 : warp - kLoaderWarp1 + 1;
        const bool lead = lq == 0;
        if (lead && lane == 0) {
            tc::prefetch_tmap(&map_q);
            if (rope) {
                tc::prefetch_tmap(&map_qr);
                tc::prefetch_tmap(&map_kr);
            }
            tc::prefetch_tmap(&map_do);
            tc::prefetch_tmap(&map_k);
            tc::prefetch_tmap(&map_v);
        }
        const int oob_row = g.t1 * g.n1;   // out of range: the TMA fills zeros
        // small groups: one box per token would be a single row, so rows are
        // fetched four at a time (tile::gather4): a load is (plane, group of 4
        // rows); otherwise (plane, token).  Load idx of a stage goes to loader
        // idx % kLoaders.
        const bool gather = G <= 4 && 4 % G == 0;
        const int per_plane = gather ? kRows / 4 : tpt;
        const uint32_t load_bytes = gather ? 4 * 128 : (uint32_t)G * 128;
        auto my_bytes = [&](int c) {
            const int first = ((lq - c * per_plane) % kLoaders + kLoaders) % kLoaders;
            return first < per_plane ? (uint32_t)((per_plane - 1 - first) / kLoaders + 1) * load_bytes : 0u;
        };
        int *ent = reinterpret_cast<int *>(smem + L::OFF_LENT) + lq * kRows;   // this warp's copy of the tile's entries
        // the loads of `planes` 64-column planes of a stage: destination plane c
        // at dst + 16 KB c, barrier bar0 + c
        auto issue = [&](const KeyTile &kt, int planes, uint8_t *dst, uint64_t *bar0, bool is_q) {
            for (int idx = lq + kLoaders * lane; idx < planes * per_plane; idx += kLoaders * 32) {
                const int c = idx / per_plane, x = idx % per_plane;
                const CUtensorMap *mp = is_q ? qmap(c) : &map_do;
                const int col = is_q ? cx(c) : c * 64;
                if (gather) {
                    // rows past the last token re-read the first token's row (their P and dS are 0)
                    int y[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = 4 * x + e, en = ent[r / G];
                        y[e] = ((en >= 0 ? en : ent[0]) / g.block_count) * g.n1 + kt.n2 * G + r % G;
                    }
                    tc::tma_gather4(dst + c * 16384 + x * 512, mp, col, y[0], y[1], y[2], y[3], bar0 + c);
                } else {
                    const int y = ent[x] >= 0 ? (ent[x] / g.block_count) * g.n1 + kt.n2 * G : oob_row;
                    tc::tma_load_2d(dst + c * 16384 + x * G * 128, mp, col, y, bar0 + c);
                }
            }
        };
        int ne = 0, tc_i = 0;
        uint32_t armed_kv = 0, armed_q[2] = {0, 0}, armed_do[2] = {0, 0};
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int64_t ti = lead ? ring_take(ring, &ws.hdr->work_counter, k, abort_flag, lane)
                                    : ring_read(ring, k, abort_flag, lane);
            if (ti < 0) { ok = false; break; }
            if (ti >= g.n_units) break;
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            if (lead) {
                if (ne > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(&bars[B_KV_EMPTY], (ne - 1) & 1, abort_flag,
                                                                       kWaitNs))) {
                    ok = false;
                    break;
                }
                ++armed_kv;
                if (lane == 0) {
                    tc::mbar_arrive_expect_tx(&bars[B_KV_FULL], (uint32_t)nk * (DQK + DV) * 2);
                    for (int c = 0; c < KC; ++c)
                        tc::tma_load_3d(smem + L::OFF_K + c * 8192, kmap(c), cx(c), kt.n2, (int)kt.key0,
                                        &bars[B_KV_FULL]);
                    for (int c = 0; c < 2; ++c)
                        tc::tma_load_3d(smem + L::OFF_V + c * 8192, &map_v, c * 64, kt.n2, (int)kt.key0,
                                        &bars[B_KV_FULL]);
                }
            }
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i & 1;
                const int nt = min(tpt, kt.ntok - i * tpt);
                // the tile's bucket entries (-1 past the last token), read
                // before waiting for the stage
                for (int tt = lane; tt < tpt; tt += 32) ent[tt] = tt < nt ? ws.entries[kt.e0 + i * tpt + tt] : -1;
                __syncwarp();
                if (tc_i >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(&bars[B_Q_EMPTY0 + s], ((tc_i >> 1) - 1) & 1,
                                                                          abort_flag, kWaitNs))) {
                    ok = false;
                    break;
                }
                if (lead) {
                    int *m = meta + (tc_i % kMeta) * kRows;
                    for (int tt = lane; tt < tpt; tt += 32) m[tt] = ent[tt];
                    __syncwarp();
                }
                ++armed_q[s];
                if (lane == 0)
                    for (int c = 0; c < KC; ++c) tc::mbar_arrive_expect_tx(&bars[B_Q_FULL + s * 3 + c], my_bytes(c));
                __syncwarp();
                issue(kt, KC, smem + L::OFF_Q + s * L::Q_STAGE, &bars[B_Q_FULL + s * 3], true);
                const int d = tc_i % DOS;
                if (tc_i >= DOS &&
                    !__all_sync(0xffffffffu, tc::mbar_wait(&bars[B_DO_EMPTY0 + d], ((tc_i / DOS) - 1) & 1, abort_flag,
                                                           kWaitNs))) {
                    ok = false;
                    break;
                }
                ++armed_do[d];
                if (lane == 0)
                    for (int c = 0; c < 2; ++c) tc::mbar_arrive_expect_tx(&bars[B_DO_FULL + d * 2 + c], my_bytes(c));
                __syncwarp();
                issue(kt, 2, smem + L::OFF_DO + d * L::DO_STAGE, &bars[B_DO_FULL + d * 2], false);
                // the entries copy is rewritten for the next tile
                __syncwarp();
            }
            ++ne;
        }
        if (!ok && lane == 0) fail();
        // let every load this warp issued land before the CTA exits
        bool drained = tc::drain_armed(&bars[B_KV_FULL], armed_kv, kWaitNs);
        for (int i = 0; i < 2; ++i) {
            for (int c = 0; c < KC; ++c)
                drained = tc::drain_armed(&bars[B_Q_FULL + i * 3 + c], armed_q[i], kWaitNs) && drained;
            for (int c = 0; c < 2; ++c)
                drained = tc::drain_armed(&bars[B_DO_FULL + i * 2 + c], armed_do[i], kWaitNs) && drained;
        }
        if (!drained) fail();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // Pipe order per query tile t:  S(t) | dK, dQ (t-1) | dP(t) | dV(t).
        // The softmax turns S(t) into P(t) while dK / dQ of t-1 and dP(t)
        // run, and dP(t) into dS(t) while dV(t) and S(t+1) run.  The whole
        // warp runs this schedule; one elected lane issues each instruction.
        const bool bf16 = !kFp16;
        const uint32_t id_s = tc::idesc_f16(kRows, nk, bf16, false, false);
        const uint32_t id_t = tc::idesc_f16(128, nk, bf16, true, true);
        const uint32_t id_q = tc::idesc_f16(kRows, DQK, bf16, false, true);
        // base descriptors; a k-step adds its byte offset / 16
        const uint64_t d_k = tc::sw128_desc(sbase + L::OFF_K, 16, 1024);      // K tile, K-major (S)
        const uint64_t d_kt = tc::sw128_desc(sbase + L::OFF_K, 8192, 1024);   // K tile, MN-major (dQ)
        const uint64_t d_v = tc::sw128_desc(sbase + L::OFF_V, 16, 1024);
        const uint64_t d_p = tc::sw128_desc(sbase + L::OFF_P, 16384, 1024);
        const uint64_t d_dst = tc::sw128_desc(sbase + L::OFF_DS, 16384, 1024);  // dS, MN-major (dK)
        const uint64_t d_dsk = tc::sw128_desc(sbase + L::OFF_DS, 16, 1024);     // dS, K-major (dQ)
        const uint64_t d_q0 = tc::sw128_desc(sbase + L::OFF_Q, 16, 1024);
        const uint64_t d_qt0 = tc::sw128_desc(sbase + L::OFF_Q, 16384, 1024);
        const uint64_t d_do0 = tc::sw128_desc(sbase + L::OFF_DO, 16, 1024);
        const uint64_t d_dot0 = tc::sw128_desc(sbase + L::OFF_DO, 16384, 1024);
        auto wait = [&](int b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, tc::mbar_wait(&bars[b], parity, abort_flag, kWaitNs));
        };
        int ne = 0, tc_i = 0;
        bool ok = true;
        // dK / dQ of tile t (local index il within its key tile)
        auto back_half = [&](int t, int il) -> bool {
            if (!wait(B_DS_FULL, t & 1)) return false;
            tc::tc_fence_after();
            const uint64_t dqt = d_qt0 + (uint64_t)(((t & 1) * L::Q_STAGE) >> 4);
            // dK^T += Q^T dS, dims [0,128) and (192 wide) dims [64,192)
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk)
                tc::mma_f16_ss_warp(tmem + kColDKlo, dqt + ((kk * 2048) >> 4), d_dst + ((kk * 2048) >> 4), id_t,
                                    (il > 0) || (kk > 0));
            if (DQK == 192) {
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk)
                    tc::mma_f16_ss_warp(tmem + kColDKhi, dqt + ((16384 + kk * 2048) >> 4), d_dst + ((kk * 2048) >> 4),
                                        id_t, (il > 0) || (kk > 0));
            }
            tc::mma_commit_warp(&bars[B_Q_EMPTY0 + (t & 1)]);
            if (!store_ds) {
                // dQ = dS K (A: dS K-major, B: K tile MN-major, N = Dqk)
                if (t > 0 && !wait(B_DQ_FREE, (t - 1) & 1)) return false;
                tc::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    if (kk < nk / 16)
                        tc::mma_f16_ss_warp(tmem + kColDQ, d_dsk + ((kk * 32) >> 4), d_kt + ((kk * 2048) >> 4), id_q,
                                            kk > 0);
            }
            tc::mma_commit_warp(&bars[B_DS_FREE]);
            tc::mma_commit_warp(&bars[B_MMA_DONE]);
            return true;
        };
        for (int k = 0; ok; ++k) {
            const int64_t ti = ring_read(ring, k, abort_flag, lane);
            if (ti < 0) { ok = false; break; }
            if (ti >= g.n_units) break;
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            if (!wait(B_KV_FULL, ne & 1)) { ok = false; break; }
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i & 1, d = tc_i % DOS;
                if (tc_i > 0 && !wait(B_S_FREE, (tc_i - 1) & 1)) { ok = false; break; }
                const uint64_t dq = d_q0 + (uint64_t)((s * L::Q_STAGE) >> 4);
                const uint64_t ddo = d_do0 + (uint64_t)((d * L::DO_STAGE) >> 4);
                const uint64_t ddot = d_dot0 + (uint64_t)((d * L::DO_STAGE) >> 4);
                // S = Q K^T (both operands K-major), chunk by chunk as they land
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk) {
                    if ((kk & 3) == 0) {
                        if (!wait(B_Q_FULL + s * 3 + (kk >> 2), (tc_i >> 1) & 1)) { ok = false; break; }
                        tc::tc_fence_after();
                    }
                    tc::mma_f16_ss_warp(tmem + kColS, dq + ((((kk >> 2) * 16384) + (kk & 3) * 32) >> 4),
                                        d_k + ((((kk >> 2) * 8192) + (kk & 3) * 32) >> 4), id_s, kk > 0);
                }
                if (!ok) break;
                tc::mma_commit_warp(&bars[B_S_FULL]);
                if (i > 0 && !back_half(tc_i - 1, i - 1)) { ok = false; break; }
                // dP = dY V^T
#pragma unroll
                for (int kk = 0; kk < DV / 16; ++kk) {
                    if ((kk & 3) == 0) {
                        if (!wait(B_DO_FULL + d * 2 + (kk >> 2), (tc_i / DOS) & 1)) { ok = false; break; }
                        tc::tc_fence_after();
                    }
                    tc::mma_f16_ss_warp(tmem + kColDP, ddo + ((((kk >> 2) * 16384) + (kk & 3) * 32) >> 4),
                                        d_v + ((((kk >> 2) * 8192) + (kk & 3) * 32) >> 4), id_s, kk > 0);
                }
                if (!ok) break;
                tc::mma_commit_warp(&bars[B_DP_FULL]);
                // dV^T += dY^T P (A: dY tile MN-major, B: P MN-major); the
                // first tile overwrites the accumulators, which the epilogue
                // must have read out for the previous key tile
                if (i == 0 && ne > 0 && !wait(B_ACC_FREE, (ne - 1) & 1)) { ok = false; break; }
                if (!wait(B_P_FULL, tc_i & 1)) { ok = false; break; }
                tc::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk)
                    tc::mma_f16_ss_warp(tmem + kColDV, ddot + ((kk * 2048) >> 4), d_p + ((kk * 2048) >> 4), id_t,
                                        (i > 0) || (kk > 0));
                tc::mma_commit_warp(&bars[B_DO_EMPTY0 + d]);
                tc::mma_commit_warp(&bars[B_P_FREE]);
            }
            if (!ok || !back_half(tc_i - 1, kt.ntiles - 1)) { ok = false; break; }
            tc::mma_commit_warp(&bars[B_ACC_FULL]);
            tc::mma_commit_warp(&bars[B_KV_EMPTY]);
            ++ne;
        }
        if (!ok && lane == 0) fail();
        // every MMA issued must be complete before TMEM is freed
        tc::mma_commit_warp(&bars[B_DRAIN]);
        if (!__all_sync(0xffffffffu, tc::mbar_wait_drain(&bars[B_DRAIN], 0, kWaitNs)) && lane == 0) fail();
    } else if (warp < 6) {
        // ------------------------------------------------------ softmax / dS
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                      // query row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const int tt = r / G, gg = r % G;
        uint8_t *prow = smem + L::OFF_P;
        uint8_t *drow = smem + L::OFF_DS;
        int tc_i = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int64_t ti = ring_read(ring, k, abort_flag, lane);
            if (ti < 0) { ok = false; break; }
            if (ti >= g.n_units) break;
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i & 1;
                ok = tc::mbar_wait(&bars[B_Q_FULL + s * 3], (tc_i >> 1) & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const int ent = tt < tpt ? meta[(tc_i % kMeta) * kRows + tt] : -1;
                const bool valid = ent >= 0;
                float lse2 = 0.f, delta = 0.f;
                if (valid) {
                    const int64_t grow = (int64_t)(ent / g.block_count) * g.n1 + kt.n2 * G + gg;
                    lse2 = ws.lse2[grow];
                    delta = ws.delta[grow];
                }
                // ---- P = exp2(S * scale * log2e - lse2): needs S only
                ok = tc::mbar_wait(&bars[B_S_FULL], tc_i & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                float pf[64];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c < nk / 16) {
                        uint32_t sv[16];
                        tc::tmem_ld16(trow + kColS + c * 16, sv);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pf[c * 16 + j] = valid ? ex2(fmaf(__uint_as_float(sv[j]), g.scale_log2, -lse2)) : 0.f;
                    }
                }
                // S is in registers: its TMEM columns may take S(t+1)
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[B_S_FREE]);
                // dV(t-1) must be done reading the P buffer
                if (tc_i > 0) {
                    ok = tc::mbar_wait(&bars[B_P_FREE], (tc_i - 1) & 1, abort_flag, kWaitNs);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (c < nk / 8)
                        *reinterpret_cast<uint4 *>(prow + sw_off(r, c)) =
                            make_uint4(pack2<kFp16>(pf[c * 8], pf[c * 8 + 1]), pack2<kFp16>(pf[c * 8 + 2], pf[c * 8 + 3]),
                                       pack2<kFp16>(pf[c * 8 + 4], pf[c * 8 + 5]), pack2<kFp16>(pf[c * 8 + 6], pf[c * 8 + 7]));
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&bars[B_P_FULL]);
                // ---- dS = P (dP - Delta)
                ok = tc::mbar_wait(&bars[B_DP_FULL], tc_i & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                uint32_t dk2[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c < nk / 16) {
                        uint32_t dv[16];
                        tc::tmem_ld16(trow + kColDP + c * 16, dv);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; j += 2)
                            dk2[c * 8 + j / 2] = pack2<kFp16>(pf[c * 16 + j] * (__uint_as_float(dv[j]) - delta),
                                                              pf[c * 16 + j + 1] * (__uint_as_float(dv[j + 1]) - delta));
                    }
                }
                // dK / dQ of t-1 must be done reading the dS buffer
                if (tc_i > 0) {
                    ok = tc::mbar_wait(&bars[B_DS_FREE], (tc_i - 1) & 1, abort_flag, kWaitNs);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (c < nk / 8)
                        *reinterpret_cast<uint4 *>(drow + sw_off(r, c)) =
                            make_uint4(dk2[c * 4], dk2[c * 4 + 1], dk2[c * 4 + 2], dk2[c * 4 + 3]);
                if (store_ds && valid) {
                    // dS[t - tok_lo][n2][slot][g][key] in the input dtype
                    const int t = ent / g.block_count, slot = ent % g.block_count;
                    const int64_t base =
                        ((((int64_t)(t - g.tok_lo) * g.n2 + kt.n2) * g.block_count + slot) * G + gg) * g.block_size +
                        kt.koff;
                    uint4 *dst = reinterpret_cast<uint4 *>(ws.ds + base);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        if (c < nk / 8) dst[c] = make_uint4(dk2[c * 4], dk2[c * 4 + 1], dk2[c * 4 + 2], dk2[c * 4 + 3]);
                }
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[B_DS_FULL]);
            }
        }
        if (!ok) fail();
    } else {
        // ------------------------------------------------------ epilogue
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const int tt = r / G, gg = r % G;
        uint8_t *stg = smem + L::OFF_STG + (warp - 6) * 4096;
        const int et = threadIdx.x - 192;                 // 0..127
        int ne = 0, tc_i = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int64_t ti = ring_read(ring, k, abort_flag, lane);
            if (ti < 0) { ok = false; break; }
            if (ti >= g.n_units) break;
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) {
                if (!g.chunked && !g.windowed) {
                    for (int i = et; i < nk * (DQK + DV); i += 128) {
                        const int j = i / (DQK + DV), c = i % (DQK + DV);
                        const int64_t row = (kt.key0 + j) * g.n2 + kt.n2;
                        if (c < DQK) *split_col(A.dk, A.dk_rope, row, c, DQK, g.d_rope) = 0;
                        else A.dv[row * DV + c - DQK] = 0;
                    }
                }
                continue;
            }
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                if (store_ds) continue;
                ok = tc::mbar_wait(&bars[B_MMA_DONE], tc_i & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                const int ent = tt < tpt ? meta[(tc_i % kMeta) * kRows + tt] : -1;
                // the tile into the fp32 accumulator (reductions) or into its
                // partial rows (stores); the choice is taken outside the loop
                auto drain = [&](auto slots) {
                    // destination row (of Dqk floats): the query row of the dQ
                    // accumulator, or the (row, slot, key tile) partial
                    int64_t grow = -1;
                    if constexpr (decltype(slots)::value) {
                        if (ent >= 0)
                            grow = (((int64_t)(ent / g.block_count - g.tok_lo) * g.n1 + kt.n2 * G + gg) *
                                        g.block_count + ent % g.block_count) * g.halves + kt.koff / nk;
                    } else {
                        grow = ent >= 0 ? (int64_t)(ent / g.block_count) * g.n1 + kt.n2 * G + gg : -1;
                    }
                    for (int c = 0; c < DQK / 32; ++c) {
                        uint32_t v0[16], v1[16];
                        tc::tmem_ld16(trow + kColDQ + c * 32, v0);
                        tc::tmem_ld16(trow + kColDQ + c * 32 + 16, v1);
                        tc::tmem_wait_ld();
                        // stage the warp's 32 rows x 32 floats, then red whole row segments
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
                        for (int k = 0; k < 8; ++k) {
                            const int rr = k * 4 + (lane >> 3), j4 = lane & 7;
                            const int64_t gr = __shfl_sync(0xffffffffu, grow, rr);
                            const float4 x = *reinterpret_cast<const float4 *>(stg + rr * 128 + ((j4 ^ (rr & 7)) << 4));
                            if (gr < 0) continue;
                            if constexpr (decltype(slots)::value)
                                __stcs(reinterpret_cast<float4 *>(ws.dq_part + gr * DQK + c * 32 + j4 * 4), x);
                            else
                                tc::red_add_v4(ws.dq_acc + gr * DQK + c * 32 + j4 * 4, x.x, x.y, x.z, x.w);
                        }
                        __syncwarp();
                    }
                };
                if (g.dq_slots) drain(std::true_type{});
                else drain(std::false_type{});
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[B_DQ_FREE]);
            }
            if (!ok) break;
            // dK / dV of this key tile
            ok = tc::mbar_wait(&bars[B_ACC_FULL], ne & 1, abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc::tc_fence_after();
            for (int j0 = 0; j0 < nk; j0 += 16) {
                uint32_t av[16], ak[16], ah[16];
                tc::tmem_ld16(trow + kColDV + j0, av);
                tc::tmem_ld16(trow + kColDKlo + j0, ak);
                if (DQK == 192) tc::tmem_ld16(trow + kColDKhi + j0, ah);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int64_t row = (kt.key0 + j0 + j) * g.n2 + kt.n2;
                    const float vv = __uint_as_float(av[j]), kv = __uint_as_float(ak[j]);
                    if (g.windowed) {
                        // partial of one token window: other windows add to the same rows
                        float *acc = ws.dkv_acc + row * (DQK + DV);
                        atomicAdd(acc + r, kv);
                        atomicAdd(acc + DQK + r, vv);
                        if (DQK == 192 && r >= 64) atomicAdd(acc + 64 + r, __uint_as_float(ah[j]));
                    } else if (g.chunked) {
                        float *acc = ws.dkv_acc + row * (DQK + DV);
                        acc[r] += kv;
                        acc[DQK + r] += vv;
                        if (DQK == 192 && r >= 64) acc[64 + r] += __uint_as_float(ah[j]);
                    } else {
                        *split_col(A.dk, A.dk_rope, row, r, DQK, g.d_rope) = f_to_u16<kFp16>(kv * g.scale);
                        A.dv[row * DV + r] = f_to_u16<kFp16>(vv);
                        if (DQK == 192 && r >= 64)
                            *split_col(A.dk, A.dk_rope, row, 64 + r, DQK, g.d_rope) =
                                f_to_u16<kFp16>(__uint_as_float(ah[j]) * g.scale);
                    }
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&bars[B_ACC_FREE]);
            ++ne;
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

}  // namespace

// G in {1, 2, 4} (rows fetched with tile::gather4): the split schedule
// measured faster there (small-group workload 19.4 -> 16.4 ms on GB300);
// SELATTN_SPLIT_SOFTMAX=0 / 1 forces the choice
bool bwd_split_preferred(const Geometry &g) {
    const char *env = getenv("SELATTN_SPLIT_SOFTMAX");
    if (env && env[0] == '0') return false;
    if (env && env[0] == '1') return true;
    return g.group <= 4 && 4 % g.group == 0;
}

template <bool kFp16, int DQK>
static cudaError_t launch_tc_t(const Geometry &g, const Workspace &ws, const sag_io &io, bool det, cudaStream_t s,
                               int num_sms) {
    const int nk = g.block_size > 64 ? 64 : g.block_size;
    TcArgs a;
    a.g = g;
    a.ws = ws;
    a.dk = (uint16_t *)io.dk;
    a.dv = (uint16_t *)io.dv;
    a.dk_rope = (uint16_t *)io.dk_rope;
    a.nk = nk;
    a.halves = g.block_size / nk;
    a.tpt = kRows / g.group;
    a.deterministic = det ? 1 : 0;
    a.n_titems = g.n_units;
    // G in {1, 2, 4}: one-row boxes for tile::gather4; otherwise one box per token (G rows)
    const uint32_t box_rows = (g.group <= 4 && 4 % g.group == 0) ? 1 : g.group;
    QkMaps m;
    CUtensorMap mdo, mv;
    if (!qk_maps(&m, g, io, kFp16, box_rows, nk) ||
        !tmap_2d(&mdo, io.attention_out_grad, kFp16, 128, (uint64_t)g.t1 * g.n1, box_rows) ||
        !tmap_3d(&mv, io.value, kFp16, 128, g.n2, g.t2, nk))
        return cudaErrorInvalidValue;
    auto fn = k_bwd_tc_split<kFp16, DQK>;
    const int smem = Smem<DQK>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int64_t grid = a.n_titems < num_sms ? a.n_titems : num_sms;
    if (grid < 1) grid = 1;
    // the launch's CTAs take their units from this counter
    if ((e = cudaMemsetAsync(&ws.hdr->work_counter, 0, sizeof(ws.hdr->work_counter), s)) != cudaSuccess) return e;
    fn<<<(int)grid, kSplitThreads, smem, s>>>(m.q, mdo, m.k, mv, m.qr, m.kr, a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_tc_split(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16,
                                bool deterministic, cudaStream_t s, int num_sms) {
    if (!bwd_tc_supported(g)) return cudaErrorInvalidValue;
    if (fp16)
        return g.d_qk == 192 ? launch_tc_t<true, 192>(g, ws, io, deterministic, s, num_sms)
                             : launch_tc_t<true, 128>(g, ws, io, deterministic, s, num_sms);
    return g.d_qk == 192 ? launch_tc_t<false, 192>(g, ws, io, deterministic, s, num_sms)
                         : launch_tc_t<false, 128>(g, ws, io, deterministic, s, num_sms);
}

}  // namespace sag
