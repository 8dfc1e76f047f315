// Tensor-core (tcgen05 / TMEM / TMA) key-block-major backward.
//
// Work unit: a key tile = NK (<= 64) consecutive key rows of one selected
// block of (batch b, KV head n2), with the bucket of (token, slot) pairs that
// selected the block ("NsaSelectedAttentionGrad" README, Gather formula,
// inverted by key block).  A persistent CTA walks its key tiles; for each it
// keeps the K / V tile in shared memory and the dK / dV accumulators in TMEM
// and streams the bucket's query rows in tiles of 128 (128 / G tokens x G
// heads).  Per query tile:
//     S    = Q K^T          (M = 128 rows, N = NK, K = Dqk)   -> TMEM
//     dP   = dY V^T         (M = 128 rows, N = NK, K = Dv)    -> TMEM
//     P    = exp2(S * scale*log2e - lse2),  dS = P (dP - Delta)  (CUDA cores)
//     dV^T += dY^T P        (M = Dv dims, N = NK, K = 128 rows)
//     dK^T += Q^T dS        (M = Dqk dims, 128 at a time, N = NK)
//     dQ   = dS K           (M = 128 rows, N = Dqk, K = NK)   -> fp32 red into
//                                                               the dQ accumulator
// (dV = P^T dY, dK = dS^T Q / sqrt(d), dQ = dS K / sqrt(d): README function
// description; dS = P * (dP - Delta): softmax adjoint of the dense formulas of
// "aclnnFlashAttentionUnpaddingScoreGradV3").  When dQ is formed by the
// fixed-order pass from the stored dS it is not formed here: dS is stored,
// and two query tiles are in flight (see the MMA role).  With per-slot
// partials each key tile's dQ tile is stored for the summing pass instead of
// being reduced.
//
// Warp roles (320 threads): 0 TMA producer, 1 MMA issuer and TMEM owner,
// 2-5 softmax / dS (thread = query row = TMEM lane), 6-9 epilogue (dQ reds per
// tile, dK / dV per key tile).  Every wait is bounded; a timeout records
// SAG_ERR_TIMEOUT and the CTA winds down.
#include "kernels.cuh"
#include "tc.cuh"
#include "tile.cuh"
#include "tmap.cuh"

namespace sag {
namespace {

constexpr int kMeta = 4;            // depth of the tile-metadata ring
constexpr int kSoftmaxWarps = 4;    // one per TMEM lane quarter
constexpr int kEpiWarp0 = 2 + kSoftmaxWarps;
constexpr int kBwdThreads = (kEpiWarp0 + 4) * 32;

// TMEM columns (512 allocated); when dS is stored the dQ columns hold a
// second S / dP set (S at kColSet1, dP at kColSet1 + 64)
constexpr uint32_t kColS = 0, kColDP = 64, kColDV = 128, kColDKlo = 192, kColDKhi = 256, kColDQ = 320;
constexpr uint32_t kColSet1 = 320;

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
    // the P and dS tiles, or, when dS is stored, the P tiles of the two query
    // tiles in flight
    static constexpr int OFF_P = OFF_DO + DOS * DO_STAGE;
    static constexpr int OFF_DS = OFF_P + 16384;
    // 4 epilogue warps x 4 KB of dQ staging, or the dS tile when dS is stored
    static constexpr int OFF_STG = OFF_DS + 16384;
    static constexpr int OFF_META = OFF_STG + 16384;     // kMeta x 128 ints
    static constexpr int OFF_BAR = OFF_META + kMeta * kRows * 4;
    static constexpr int TOTAL = OFF_BAR + 256 + 1024;   // + slack for 1024-B alignment
};

enum Bar {
    B_KV_FULL = 0, B_KV_EMPTY, B_Q_FULL0, B_Q_FULL1, B_Q_EMPTY0, B_Q_EMPTY1, B_DO_FULL0, B_DO_FULL1,
    B_DO_EMPTY0, B_DO_EMPTY1, B_S_FULL, B_S_FULL1, B_DP_FULL, B_DP_FULL1, B_P_FULL, B_DS_FULL,
    B_MMA_DONE, B_MMA_DONE1, B_DQ_FREE, B_ACC_FULL, B_ACC_FREE, B_DRAIN, B_COUNT
};

struct TcArgs {
    Geometry g;
    Workspace ws;
    uint16_t *dk, *dv, *dk_rope;
    int nk, halves, tpt, deterministic;
    int early_s;            // issue S = Q K^T before dY has landed (one tile in flight)
    int64_t n_titems;
};

// dQ modes of a launch (compile-time, so each mode's loops carry no branch
// for the others): reductions into the fp32 accumulator, dS stored for the
// fixed-order pass, or per-slot fp32 partials for the summing pass
enum DqMode { kDqRed = 0, kDqStoreDs = 1, kDqSlots = 2 };

template <bool kFp16, int DQK, int kMode>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_bwd_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
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
    // fixed-order dQ: from the stored dS (a later pass re-reads the key
    // blocks), or from per-slot fp32 partials of dQ = dS K stored here
    constexpr bool store_ds = kMode == kDqStoreDs;
    // the whole MMA warp runs the schedule when dS is stored (see the MMA role)
    constexpr bool kWarpIssue = kMode == kDqStoreDs;
    // when dS is stored, two query tiles are in flight (see the MMA role);
    // otherwise one tile at a time, P and dS handed over at once
    constexpr bool kPipelined = kMode == kDqStoreDs;
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
            tc::mbar_init(&bars[B_Q_FULL0 + s], 1);
            tc::mbar_init(&bars[B_Q_EMPTY0 + s], 1);
            tc::mbar_init(&bars[B_DO_FULL0 + s], 1);
            tc::mbar_init(&bars[B_DO_EMPTY0 + s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&bars[B_S_FULL + b], 1);
            tc::mbar_init(&bars[B_DP_FULL + b], 1);
            tc::mbar_init(&bars[B_MMA_DONE + b], 1);
        }
        tc::mbar_init(&bars[B_P_FULL], kSoftmaxWarps * 32);
        tc::mbar_init(&bars[B_DS_FULL], kSoftmaxWarps * 32);
        tc::mbar_init(&bars[B_DQ_FREE], 128);
        tc::mbar_init(&bars[B_ACC_FULL], 1);
        tc::mbar_init(&bars[B_ACC_FREE], 128);
        tc::mbar_init(&bars[B_DRAIN], 1);
        tc::fence_mbar_init();
    }
    // rows of a Q / dY tile no token fills (when G does not divide 128) must
    // hold finite values: zero the staging buffers once
    if (tpt * G < kRows) {
        for (int i = threadIdx.x; i < (2 * L::Q_STAGE + DOS * L::DO_STAGE) / 16; i += kBwdThreads)
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

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::prefetch_tmap(&map_q);
            tc::prefetch_tmap(&map_do);
            tc::prefetch_tmap(&map_k);
            tc::prefetch_tmap(&map_v);
            if (rope) {
                tc::prefetch_tmap(&map_qr);
                tc::prefetch_tmap(&map_kr);
            }
        }
        const int oob_row = g.t1 * g.n1;   // out of range: the TMA fills zeros
        // small groups: one box per token would be a single row, so rows are
        // fetched four at a time (tile::gather4) instead
        const bool gather = G <= 4 && 4 % G == 0;
        int ne = 0, tc_i = 0;
        uint32_t armed_kv = 0, armed_q[2] = {0, 0}, armed_do[2] = {0, 0};
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            if (ne > 0 && !tc::mbar_wait(&bars[B_KV_EMPTY], (ne - 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            ++armed_kv;
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(&bars[B_KV_FULL], (uint32_t)nk * (DQK + DV) * 2);
                for (int c = 0; c < KC; ++c)
                    tc::tma_load_3d(smem + L::OFF_K + c * 8192, kmap(c), cx(c), kt.n2, (int)kt.key0, &bars[B_KV_FULL]);
                for (int c = 0; c < 2; ++c)
                    tc::tma_load_3d(smem + L::OFF_V + c * 8192, &map_v, c * 64, kt.n2, (int)kt.key0, &bars[B_KV_FULL]);
            }
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i & 1;
                const int nt = min(tpt, kt.ntok - i * tpt);
                // the tile's bucket entries (up to 128 tokens: 4 per lane), loaded
                // before waiting for the stage
                int ent[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int tt = lane + 32 * q;
                    ent[q] = tt < nt ? ws.entries[kt.e0 + i * tpt + tt] : -1;
                }
                if (tc_i >= 2 && !tc::mbar_wait(&bars[B_Q_EMPTY0 + s], ((tc_i >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                int *m = meta + (tc_i % kMeta) * kRows;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (lane + 32 * q < tpt) m[lane + 32 * q] = ent[q];
                __syncwarp();
                ++armed_q[s];
                if (lane == 0) tc::mbar_arrive_expect_tx(&bars[B_Q_FULL0 + s], (uint32_t)tpt * G * DQK * 2);
                __syncwarp();
                uint8_t *qdst = smem + L::OFF_Q + s * L::Q_STAGE;
                if (gather) {
                    // G in {1, 2, 4}: lane k fetches tile rows 4k..4k+3 with one gather4 per chunk
                    int y[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = 4 * lane + j, tk = row / G;
                        // rows past the last token re-read the first token's row (their P and dS are 0)
                        y[j] = (m[tk < nt ? tk : 0] / g.block_count) * g.n1 + kt.n2 * G + row % G;
                    }
                    for (int c = 0; c < KC; ++c)
                        tc::tma_gather4(qdst + c * 16384 + lane * 512, qmap(c), cx(c), y[0], y[1], y[2], y[3],
                                        &bars[B_Q_FULL0 + s]);
                } else {
                    // one (token, chunk) box per lane: the issue is spread over the warp
                    for (int j = lane; j < tpt * KC; j += 32) {
                        const int tt = j / KC, c = j % KC;
                        const int y = tt < nt ? (m[tt] / g.block_count) * g.n1 + kt.n2 * G : oob_row;
                        tc::tma_load_2d(qdst + c * 16384 + tt * G * 128, qmap(c), cx(c), y, &bars[B_Q_FULL0 + s]);
                    }
                }
                const int d = tc_i % DOS;
                if (tc_i >= DOS &&
                    !tc::mbar_wait(&bars[B_DO_EMPTY0 + d], ((tc_i / DOS) - 1) & 1, abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                ++armed_do[d];
                if (lane == 0) tc::mbar_arrive_expect_tx(&bars[B_DO_FULL0 + d], (uint32_t)tpt * G * DV * 2);
                __syncwarp();
                uint8_t *ddst = smem + L::OFF_DO + d * L::DO_STAGE;
                if (gather) {
                    int y[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = 4 * lane + j, tk = row / G;
                        // rows past the last token re-read the first token's row (their P and dS are 0)
                        y[j] = (m[tk < nt ? tk : 0] / g.block_count) * g.n1 + kt.n2 * G + row % G;
                    }
                    for (int c = 0; c < 2; ++c)
                        tc::tma_gather4(ddst + c * 16384 + lane * 512, &map_do, c * 64, y[0], y[1], y[2], y[3],
                                        &bars[B_DO_FULL0 + d]);
                } else {
                    for (int j = lane; j < tpt * 2; j += 32) {
                        const int tt = j / 2, c = j % 2;
                        const int y = tt < nt ? (m[tt] / g.block_count) * g.n1 + kt.n2 * G : oob_row;
                        tc::tma_load_2d(ddst + c * 16384 + tt * G * 128, &map_do, c * 64, y, &bars[B_DO_FULL0 + d]);
                    }
                }
            }
            ++ne;
        }
        if (!ok) fail();
        // let every load this warp issued land before the CTA exits
        bool drained = tc::drain_armed(&bars[B_KV_FULL], armed_kv, kWaitNs);
        for (int i = 0; i < 2; ++i)
            drained = tc::drain_armed(&bars[B_Q_FULL0 + i], armed_q[i], kWaitNs) &&
                      tc::drain_armed(&bars[B_DO_FULL0 + i], armed_do[i], kWaitNs) && drained;
        if (!drained) fail();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // With kWarpIssue the whole warp runs the schedule and one elected
        // lane issues each instruction, else lane 0 alone runs it: measured on
        // GB300, the warp form is faster in the deterministic mode (long
        // context 15.35 -> 14.80 ms, max selection 1358 -> 1266 ms) and slower
        // with the per-tile dQ reductions (9.93 -> 10.45 ms, 961 -> 1031 ms).
        if (kWarpIssue || lane == 0) {
        const bool bf16 = !kFp16;
        const uint32_t id_s = tc::idesc_f16(kRows, nk, bf16, false, false);
        const uint32_t id_t = tc::idesc_f16(128, nk, bf16, true, true);
        const uint32_t id_q = tc::idesc_f16(kRows, DQK, bf16, false, true);
        const uint32_t ks = sbase + L::OFF_K, vs = sbase + L::OFF_V;
        const uint32_t ps = sbase + L::OFF_P, dss = sbase + L::OFF_DS;
        auto wait = [&](int b, uint32_t parity) -> bool {
            const bool w = tc::mbar_wait(&bars[b], parity, abort_flag, kWaitNs);
            return kWarpIssue ? __all_sync(0xffffffffu, w) : w;
        };
        auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
            if (kWarpIssue) tc::mma_f16_ss_warp(d, a, b, id, acc);
            else tc::mma_f16_ss(d, a, b, id, acc);
        };
        auto commit = [&](uint64_t *bar) {
            if (kWarpIssue) tc::mma_commit_warp(bar);
            else tc::mma_commit(bar);
        };
        int ne = 0, tc_i = 0;
        bool ok = true;
        if constexpr (kPipelined) {
            // Two query tiles in flight.  Tile t has TMEM set t & 1 for S / dP
            // and shared tile t & 1 for P; dS has one shared tile (the dQ
            // staging area, unused here).  Per tile t: dV(t) once P(t) has
            // landed, S(t+1), dK(t) once dS(t) has landed, dP(t+1); the
            // softmax forms P(t+1) while dK(t) and dP(t+1) run.  Set t & 1 is
            // free for S(t+2) once dS(t) has landed (the softmax has loaded
            // dP(t) by then); the dS tile is free for dS(t+1) once dP(t+1) has
            // completed, since dK(t) was issued before it.  Tiles of one key
            // tile only: the next key tile's K / V wait for this one's MMAs.
            auto set_col = [](int t) { return (t & 1) ? kColSet1 : 0u; };
            auto issue_s = [&](int t) -> bool {
                const int st = t & 1;
                if (!wait(B_Q_FULL0 + st, (t >> 1) & 1)) return false;
                tc::tc_fence_after();
                const uint32_t qs = sbase + L::OFF_Q + st * L::Q_STAGE;
                for (int kk = 0; kk < DQK / 16; ++kk)
                    mma(tmem + set_col(t) + kColS, tc::sw128_desc(qs + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                        tc::sw128_desc(ks + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
                commit(&bars[B_S_FULL + st]);
                return true;
            };
            auto issue_dp = [&](int t) -> bool {
                const int d = t % DOS;
                if (!wait(B_DO_FULL0 + d, (t / DOS) & 1)) return false;
                tc::tc_fence_after();
                const uint32_t ds_ = sbase + L::OFF_DO + d * L::DO_STAGE;
                for (int kk = 0; kk < DV / 16; ++kk)
                    mma(tmem + set_col(t) + kColDP, tc::sw128_desc(ds_ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                        tc::sw128_desc(vs + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
                commit(&bars[B_DP_FULL + (t & 1)]);
                return true;
            };
            for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
                const KeyTile kt = decode(g, ws, ti, nk, tpt);
                if (kt.ntok == 0) continue;
                if (!wait(B_KV_FULL, ne & 1)) { ok = false; break; }
                if (ne > 0 && !wait(B_ACC_FREE, (ne - 1) & 1)) { ok = false; break; }
                if (!issue_s(tc_i) || !issue_dp(tc_i)) { ok = false; break; }
                for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                    const int s = tc_i & 1, d = tc_i % DOS;
                    const bool more = i + 1 < kt.ntiles;
                    const uint32_t qs = sbase + L::OFF_Q + s * L::Q_STAGE;
                    const uint32_t ds_ = sbase + L::OFF_DO + d * L::DO_STAGE;
                    const uint32_t pt = s ? dss : ps, dst_s = sbase + L::OFF_STG;
                    if (!wait(B_P_FULL, tc_i & 1)) { ok = false; break; }
                    tc::tc_fence_after();
                    // dV^T += dY^T P (A: dY tile MN-major, B: P MN-major)
                    for (int kk = 0; kk < kRows / 16; ++kk)
                        mma(tmem + kColDV, tc::sw128_desc(ds_ + kk * 2048, 16384, 1024),
                            tc::sw128_desc(pt + kk * 2048, 16384, 1024), id_t, (i > 0) || (kk > 0));
                    commit(&bars[B_DO_EMPTY0 + d]);
                    if (more && !issue_s(tc_i + 1)) { ok = false; break; }
                    if (!wait(B_DS_FULL, tc_i & 1)) { ok = false; break; }
                    tc::tc_fence_after();
                    // dK^T += Q^T dS, dims [0,128) and (192 wide) dims [64,192)
                    for (int kk = 0; kk < kRows / 16; ++kk)
                        mma(tmem + kColDKlo, tc::sw128_desc(qs + kk * 2048, 16384, 1024),
                            tc::sw128_desc(dst_s + kk * 2048, 16384, 1024), id_t, (i > 0) || (kk > 0));
                    if (DQK == 192)
                        for (int kk = 0; kk < kRows / 16; ++kk)
                            mma(tmem + kColDKhi, tc::sw128_desc(qs + 16384 + kk * 2048, 16384, 1024),
                                tc::sw128_desc(dst_s + kk * 2048, 16384, 1024), id_t, (i > 0) || (kk > 0));
                    commit(&bars[B_Q_EMPTY0 + s]);
                    commit(&bars[B_MMA_DONE + s]);
                    if (more && !issue_dp(tc_i + 1)) { ok = false; break; }
                }
                if (!ok) break;
                commit(&bars[B_ACC_FULL]);
                commit(&bars[B_KV_EMPTY]);
                ++ne;
            }
        } else {
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            if (!wait(B_KV_FULL, ne & 1)) { ok = false; break; }
            if (ne > 0 && !wait(B_ACC_FREE, (ne - 1) & 1)) { ok = false; break; }
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i & 1, d = tc_i % DOS;
                if (!wait(B_Q_FULL0 + s, (tc_i >> 1) & 1) ||
                    (!A.early_s && !wait(B_DO_FULL0 + d, (tc_i / DOS) & 1))) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t qs = sbase + L::OFF_Q + s * L::Q_STAGE;
                const uint32_t ds_ = sbase + L::OFF_DO + d * L::DO_STAGE;
                // S = Q K^T, dP = dY V^T (both operands K-major); with early_s
                // S is issued before dY has landed
                for (int kk = 0; kk < DQK / 16; ++kk)
                    mma(tmem + kColS, tc::sw128_desc(qs + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                        tc::sw128_desc(ks + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
                if (A.early_s && !wait(B_DO_FULL0 + d, (tc_i / DOS) & 1)) { ok = false; break; }
                tc::tc_fence_after();
                for (int kk = 0; kk < DV / 16; ++kk)
                    mma(tmem + kColDP, tc::sw128_desc(ds_ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                        tc::sw128_desc(vs + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
                commit(&bars[B_S_FULL]);
                if (!wait(B_P_FULL, tc_i & 1)) { ok = false; break; }
                tc::tc_fence_after();
                // dV^T += dY^T P (A: dY tile MN-major, B: P MN-major)
                for (int kk = 0; kk < kRows / 16; ++kk)
                    mma(tmem + kColDV, tc::sw128_desc(ds_ + kk * 2048, 16384, 1024),
                        tc::sw128_desc(ps + kk * 2048, 16384, 1024), id_t, (i > 0) || (kk > 0));
                commit(&bars[B_DO_EMPTY0 + d]);
                // dK^T += Q^T dS, dims [0,128) and (192 wide) dims [64,192)
                for (int kk = 0; kk < kRows / 16; ++kk)
                    mma(tmem + kColDKlo, tc::sw128_desc(qs + kk * 2048, 16384, 1024),
                        tc::sw128_desc(dss + kk * 2048, 16384, 1024), id_t, (i > 0) || (kk > 0));
                if (DQK == 192)
                    for (int kk = 0; kk < kRows / 16; ++kk)
                        mma(tmem + kColDKhi, tc::sw128_desc(qs + 16384 + kk * 2048, 16384, 1024),
                            tc::sw128_desc(dss + kk * 2048, 16384, 1024), id_t, (i > 0) || (kk > 0));
                commit(&bars[B_Q_EMPTY0 + s]);
                // dQ = dS K (A: dS K-major, B: K tile MN-major, N = Dqk)
                if (tc_i > 0 && !wait(B_DQ_FREE, (tc_i - 1) & 1)) { ok = false; break; }
                tc::tc_fence_after();
                for (int kk = 0; kk < nk / 16; ++kk)
                    mma(tmem + kColDQ, tc::sw128_desc(dss + kk * 32, 16, 1024),
                        tc::sw128_desc(ks + kk * 2048, 8192, 1024), id_q, kk > 0);
                commit(&bars[B_MMA_DONE]);
            }
            if (!ok) break;
            commit(&bars[B_ACC_FULL]);
            commit(&bars[B_KV_EMPTY]);
            ++ne;
        }
        }
        if (!ok && lane == 0) fail();
        // every MMA issued must be complete before TMEM is freed
        commit(&bars[B_DRAIN]);
        const bool drained = tc::mbar_wait_drain(&bars[B_DRAIN], 0, kWaitNs);
        if (!(kWarpIssue ? __all_sync(0xffffffffu, drained) : drained) && lane == 0) fail();
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------ softmax / dS
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                      // query row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const int tt = r / G, gg = r % G;
        int tc_i = 0;
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i & 1;
                ok = tc::mbar_wait(&bars[B_Q_FULL0 + s], (tc_i >> 1) & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const int ent = tt < tpt ? meta[(tc_i % kMeta) * kRows + tt] : -1;
                const bool valid = ent >= 0;
                int64_t grow = 0;
                float lse2 = 0.f, delta = 0.f;
                if (valid) {
                    grow = (int64_t)(ent / g.block_count) * g.n1 + kt.n2 * G + gg;
                    lse2 = ws.lse2[grow];
                    delta = ws.delta[grow];
                }
                if constexpr (kPipelined)
                    ok = tc::mbar_wait(&bars[B_S_FULL + s], (tc_i >> 1) & 1, abort_flag, kWaitNs);
                else
                    ok = tc::mbar_wait(&bars[B_S_FULL], tc_i & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                uint8_t *prow = smem + L::OFF_P;
                uint8_t *drow = smem + L::OFF_DS;
                if constexpr (kPipelined) {
                    // this tile's S / dP set and P tile; the one dS tile
                    uint8_t *buf = s ? drow : prow;
                    uint8_t *dsb = smem + L::OFF_STG;
                    const uint32_t tset = trow + (s ? kColSet1 : 0u);
                    // the MMAs two tiles back must be done with the P tile (they
                    // are: S of this tile was issued after them)
                    if (tc_i >= 2) {
                        ok = tc::mbar_wait(&bars[B_MMA_DONE + s], ((tc_i >> 1) - 1) & 1, abort_flag, kWaitNs);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    }
                    // dS[t - tok_lo][n2][slot][g][key] in the input dtype
                    uint4 *dst = nullptr;
                    if (valid) {
                        const int t = ent / g.block_count, slot = ent % g.block_count;
                        dst = reinterpret_cast<uint4 *>(
                            ws.ds + ((((int64_t)(t - g.tok_lo) * g.n2 + kt.n2) * g.block_count + slot) * G + gg) *
                                        g.block_size + kt.koff);
                    }
                    // P from S in two rounds of 32 keys, each round's loads in
                    // flight before one wait; P stays in fp32 for dS
                    float pf[64];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (32 * h >= nk) break;
                        uint32_t sv[4][8];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (32 * h + 8 * j < nk) tc::tmem_ld8(tset + kColS + 32 * h + 8 * j, sv[j]);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (32 * h + 8 * j >= nk) break;
                            uint32_t pk[4];
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const int k = 32 * h + 8 * j + e;
                                float p0 = 0.f, p1 = 0.f;
                                if (valid) {
                                    p0 = ex2(fmaf(__uint_as_float(sv[j][e]), g.scale_log2, -lse2));
                                    p1 = ex2(fmaf(__uint_as_float(sv[j][e + 1]), g.scale_log2, -lse2));
                                }
                                pf[k] = p0;
                                pf[k + 1] = p1;
                                pk[e / 2] = pack2<kFp16>(p0, p1);
                            }
                            *reinterpret_cast<uint4 *>(buf + sw_off(r, 4 * h + j)) =
                                make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                    tc::fence_proxy_async_smem();
                    tc::tc_fence_before();
                    tc::mbar_arrive(&bars[B_P_FULL]);
                    // dS = P (dP - Delta) once dP has landed (dK of the previous
                    // tile, issued before dP, is then done with the dS tile),
                    // also to the workspace
                    ok = tc::mbar_wait(&bars[B_DP_FULL + s], (tc_i >> 1) & 1, abort_flag, kWaitNs);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc::tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (32 * h >= nk) break;
                        uint32_t dv[4][8];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (32 * h + 8 * j < nk) tc::tmem_ld8(tset + kColDP + 32 * h + 8 * j, dv[j]);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (32 * h + 8 * j >= nk) break;
                            uint32_t w4[4];
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const int k = 32 * h + 8 * j + e;
                                float d0 = 0.f, d1 = 0.f;
                                if (valid) {
                                    d0 = pf[k] * (__uint_as_float(dv[j][e]) - delta);
                                    d1 = pf[k + 1] * (__uint_as_float(dv[j][e + 1]) - delta);
                                }
                                w4[e / 2] = pack2<kFp16>(d0, d1);
                            }
                            const uint4 v4 = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            *reinterpret_cast<uint4 *>(dsb + sw_off(r, 4 * h + j)) = v4;
                            if (valid) dst[4 * h + j] = v4;
                        }
                    }
                    tc::fence_proxy_async_smem();
                    tc::tc_fence_before();
                    tc::mbar_arrive(&bars[B_DS_FULL]);
                } else {
                    // S and dP in two rounds of 32 keys, each round's loads in
                    // flight before one wait
                    uint32_t pk[32], dk2[32];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (32 * h >= nk) break;
                        uint32_t sv[4][8], dv[4][8];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (32 * h + 8 * j < nk) {
                                tc::tmem_ld8(trow + kColS + 32 * h + 8 * j, sv[j]);
                                tc::tmem_ld8(trow + kColDP + 32 * h + 8 * j, dv[j]);
                            }
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (32 * h + 8 * j >= nk) break;
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                float p0 = 0.f, p1 = 0.f, d0 = 0.f, d1 = 0.f;
                                if (valid) {
                                    p0 = ex2(fmaf(__uint_as_float(sv[j][e]), g.scale_log2, -lse2));
                                    p1 = ex2(fmaf(__uint_as_float(sv[j][e + 1]), g.scale_log2, -lse2));
                                    d0 = p0 * (__uint_as_float(dv[j][e]) - delta);
                                    d1 = p1 * (__uint_as_float(dv[j][e + 1]) - delta);
                                }
                                pk[16 * h + j * 4 + e / 2] = pack2<kFp16>(p0, p1);
                                dk2[16 * h + j * 4 + e / 2] = pack2<kFp16>(d0, d1);
                            }
                        }
                    }
                    // the previous tile's MMAs must be done with the P / dS buffers
                    if (tc_i > 0) {
                        ok = tc::mbar_wait(&bars[B_MMA_DONE], (tc_i - 1) & 1, abort_flag, kWaitNs);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (8 * j >= nk) break;
                        *reinterpret_cast<uint4 *>(prow + sw_off(r, j)) =
                            make_uint4(pk[j * 4], pk[j * 4 + 1], pk[j * 4 + 2], pk[j * 4 + 3]);
                        *reinterpret_cast<uint4 *>(drow + sw_off(r, j)) =
                            make_uint4(dk2[j * 4], dk2[j * 4 + 1], dk2[j * 4 + 2], dk2[j * 4 + 3]);
                    }
                    tc::fence_proxy_async_smem();
                    tc::tc_fence_before();
                    tc::mbar_arrive(&bars[B_P_FULL]);
                }
            }
        }
        if (!ok) fail();
    } else {
        // ------------------------------------------------------ epilogue
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const int tt = r / G, gg = r % G;
        uint8_t *stg = smem + L::OFF_STG + (warp - kEpiWarp0) * 4096;
        const int et = threadIdx.x - kEpiWarp0 * 32;      // 0..127
        int ne = 0, tc_i = 0;
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
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
                // destination row (of Dqk floats): the query row of the dQ
                // accumulator, or the (row, slot, key tile) partial
                int64_t grow = -1;
                if constexpr (kMode == kDqSlots) {
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
                        if constexpr (kMode == kDqSlots) {
                            if (gr >= 0) __stcs(reinterpret_cast<float4 *>(ws.dq_part + gr * DQK + c * 32 + j4 * 4), x);
                        } else {
                            if (gr >= 0) tc::red_add_v4(ws.dq_acc + gr * DQK + c * 32 + j4 * 4, x.x, x.y, x.z, x.w);
                        }
                    }
                    __syncwarp();
                }
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

bool bwd_tc_supported(const Geometry &g) {
    const int bs = g.block_size;
    return g.d_v == 128 && (g.d_qk == 128 || g.d_qk == 192) &&
           (bs == 16 || bs == 32 || bs == 48 || bs == 64 || bs == 128);
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
    // S ahead of dY: measured on GB300 faster in the deterministic mode and for
    // G >= 32 (max selection 1001 -> 961 ms, long context deterministic
    // 16.0 -> 15.2 ms), slower for the default mode at G = 16 (long context
    // 10.45 -> 10.87 ms)
    a.early_s = (det || g.group >= 32) ? 1 : 0;
    a.n_titems = g.n_units;
    // G in {1, 2, 4}: one-row boxes for tile::gather4; otherwise one box per token (G rows)
    const uint32_t box_rows = (g.group <= 4 && 4 % g.group == 0) ? 1 : g.group;
    QkMaps m;
    CUtensorMap mdo, mv;
    if (!qk_maps(&m, g, io, kFp16, box_rows, nk) ||
        !tmap_2d(&mdo, io.attention_out_grad, kFp16, 128, (uint64_t)g.t1 * g.n1, box_rows) ||
        !tmap_3d(&mv, io.value, kFp16, 128, g.n2, g.t2, nk))
        return cudaErrorInvalidValue;
    auto fn = !det ? k_bwd_tc<kFp16, DQK, kDqRed>
              : g.dq_slots ? k_bwd_tc<kFp16, DQK, kDqSlots> : k_bwd_tc<kFp16, DQK, kDqStoreDs>;
    const int smem = Smem<DQK>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int64_t grid = a.n_titems < num_sms ? a.n_titems : num_sms;
    if (grid < 1) grid = 1;
    fn<<<(int)grid, kBwdThreads, smem, s>>>(m.q, mdo, m.k, mv, m.qr, m.kr, a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_tc(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, bool deterministic,
                          cudaStream_t s, int num_sms) {
    if (!bwd_tc_supported(g)) return cudaErrorInvalidValue;
    if (fp16)
        return g.d_qk == 192 ? launch_tc_t<true, 192>(g, ws, io, deterministic, s, num_sms)
                             : launch_tc_t<true, 128>(g, ws, io, deterministic, s, num_sms);
    return g.d_qk == 192 ? launch_tc_t<false, 192>(g, ws, io, deterministic, s, num_sms)
                         : launch_tc_t<false, 128>(g, ws, io, deterministic, s, num_sms);
}

}  // namespace sag
