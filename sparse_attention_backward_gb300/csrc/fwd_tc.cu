// Tensor-core (tcgen05 / TMEM / TMA) forward of selected attention, walking
// the same key tiles of the inverted index as the backward, in two passes:
//   pass 1   S = Q K^T per key tile; the row maximum of scale*S goes to m
//            (order-preserving float atomic max, exact in any order)
//   pass 2   P = exp(scale*S - m); row sums of P go to l (fp32 atomics) and
//            O += P V (M = 128 rows, N = Dv, K = keys) goes to an fp32
//            accumulator with warp-coalesced reductions
//   finalize O = O_acc / l in the input dtype; softmaxMax = m and
//            softmaxSum = l written to the 8 lanes of [T1, N1, 8]
// This is softmax(scale Q Ksel^T) Vsel over the gathered rows ("NsaSelected-
// AttentionGrad" README, function description and Gather formula; forward
// formula of "aclnnFlashAttentionUnpaddingScoreGradV3"), producing the
// attentionOut, softmaxMax and softmaxSum the backward takes as inputs (same
// README, parameter table).  The maxima are exact; the sums and O depend on
// the order of the fp32 additions (not bitwise reproducible).
//
// Warp roles as in the backward: 0 TMA producer (K / V per key tile, Q per
// query tile, three Q stages), 1 MMA issuer and TMEM owner, 2-5 softmax
// (thread = query row = TMEM lane), 6-9 O drain (pass 2), 10 second Q loader
// (odd 64-column planes: one warp issues a tile::gather4 about every 66
// cycles, so a single warp would bound the small-group tiles).
#include "kernels.cuh"
#include "tc.cuh"
#include "tile.cuh"
#include "tmap.cuh"

namespace sag {
namespace {

constexpr int kQStages = 3;
constexpr int kFwdLoader2 = 10;
constexpr int kFwdThreads = (kFwdLoader2 + 1) * 32;
constexpr int kMetaF = 8;                    // tile-metadata ring depth
constexpr uint32_t kColS = 0, kColO = 128;   // TMEM columns (256 allocated)

template <int DQK>
struct FwdSmem {
    static constexpr int KC = DQK / 64;
    static constexpr int K_TILE = KC * 8192;
    static constexpr int V_TILE = 2 * 8192;
    static constexpr int Q_STAGE = KC * 16384;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + K_TILE;
    static constexpr int OFF_Q = OFF_V + V_TILE;
    static constexpr int OFF_P = OFF_Q + kQStages * Q_STAGE;
    static constexpr int OFF_STG = OFF_P + 16384;       // 4 drain warps x 4 KB
    static constexpr int OFF_META = OFF_STG + 16384;    // kMetaF x 128 ints
    static constexpr int OFF_BAR = OFF_META + kMetaF * kRows * 4;
    static constexpr int TOTAL = OFF_BAR + 256 + 1024;  // + slack for 1024-B alignment
};

// S_FULL: S in TMEM; P_FULL: the softmax is done with S (and, in pass 2, P is
// in shared memory); O_DONE: the P V MMAs of a tile are done; O_FREE: drained.
enum FBar {
    F_KV_FULL = 0, F_KV_EMPTY, F_Q_FULL, F_Q_EMPTY = F_Q_FULL + kQStages, F_S_FULL = F_Q_EMPTY + kQStages,
    F_P_FULL, F_O_DONE, F_O_FREE, F_DRAIN, F_COUNT
};

struct FwdArgs {
    Geometry g;
    Workspace ws;
    int nk, tpt;
};

// max over any order of updates; all values finite (m starts at -inf)
__device__ __forceinline__ void atomic_max_f32(float *addr, float v) {
    if (v >= 0.f) atomicMax(reinterpret_cast<int *>(addr), __float_as_int(v));
    else atomicMin(reinterpret_cast<unsigned int *>(addr), __float_as_uint(v));
}

template <bool kFp16, int DQK, int PASS>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
             const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_qr,
             const __grid_constant__ CUtensorMap map_kr, FwdArgs A) {
    using L = FwdSmem<DQK>;
    constexpr int DV = 128;
    constexpr int KC = L::KC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_BAR + 8 * F_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_BAR + 8 * F_COUNT + 4);
    int *meta = reinterpret_cast<int *>(smem + L::OFF_META);
    const Geometry &g = A.g;
    const Workspace &ws = A.ws;
    float *mrow = ws.lse2;     // row maxima of scale * S
    float *lrow = ws.delta;    // row sums of P
    float *oacc = ws.dq_acc;   // [T1 * n1, Dv] fp32
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = A.nk, tpt = A.tpt, G = g.group;
    const uint32_t sbase = tc::smem_u32(smem);
    // 64-column chunk c of a q / k row: the main tensor at column 64 c, or
    // with the rope split chunk 2 from the rope tensor at column 0
    const bool rope = g.d_rope != 0;
    auto qmap = [&](int c) { return (rope && c == 2) ? &map_qr : &map_q; };
    auto kmap = [&](int c) { return (rope && c == 2) ? &map_kr : &map_k; };
    auto cx = [&](int c) { return (rope && c == 2) ? 0 : c * 64; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        tc::mbar_init(&bars[F_KV_FULL], 1);
        tc::mbar_init(&bars[F_KV_EMPTY], 1);
        for (int s = 0; s < kQStages; ++s) {
            tc::mbar_init(&bars[F_Q_FULL + s], 2);   // the two Q loaders
            tc::mbar_init(&bars[F_Q_EMPTY + s], 1);
        }
        tc::mbar_init(&bars[F_S_FULL], 1);
        tc::mbar_init(&bars[F_P_FULL], 128);
        tc::mbar_init(&bars[F_O_DONE], 1);
        tc::mbar_init(&bars[F_O_FREE], 128);
        tc::mbar_init(&bars[F_DRAIN], 1);
        tc::fence_mbar_init();
    }
    // rows of a Q tile no token fills (when G does not divide 128) must hold
    // finite values: zero the stages once
    if (tpt * G < kRows) {
        for (int i = threadIdx.x; i < kQStages * L::Q_STAGE / 16; i += kFwdThreads)
            reinterpret_cast<uint4 *>(smem + L::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
        tc::fence_proxy_async_smem();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 256);
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

    if (warp == 0 || warp == kFwdLoader2) {
        // ------------------------------------------------------ TMA producers
        // Warp 0 loads K / V, writes the tile metadata and the even 64-column
        // planes of each Q tile; warp 10 the odd planes.  Each arms the Q
        // stage barrier (two arrivals) with its own bytes.
        const bool lead = warp == 0;
        const int lq = lead ? 0 : 1;
        if (lead && lane == 0) {
            tc::prefetch_tmap(&map_q);
            tc::prefetch_tmap(&map_k);
            if (rope) {
                tc::prefetch_tmap(&map_qr);
                tc::prefetch_tmap(&map_kr);
            }
            if (PASS == 2) tc::prefetch_tmap(&map_v);
        }
        const int oob_row = g.t1 * g.n1;   // out of range: the TMA fills zeros
        const bool gather = G <= 4 && 4 % G == 0;
        const int my_planes = (KC - lq + 1) / 2;   // planes lq, lq + 2, ...
        int ne = 0, tc_i = 0;
        uint32_t armed_kv = 0, armed_q[kQStages] = {};
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            if (lead) {
                if (ne > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(&bars[F_KV_EMPTY], (ne - 1) & 1, abort_flag,
                                                                       kWaitNs))) {
                    ok = false;
                    break;
                }
                ++armed_kv;
                if (lane == 0) {
                    tc::mbar_arrive_expect_tx(&bars[F_KV_FULL], (uint32_t)nk * (DQK + (PASS == 2 ? DV : 0)) * 2);
                    for (int c = 0; c < KC; ++c)
                        tc::tma_load_3d(smem + L::OFF_K + c * 8192, kmap(c), cx(c), kt.n2, (int)kt.key0,
                                        &bars[F_KV_FULL]);
                    if (PASS == 2)
                        for (int c = 0; c < 2; ++c)
                            tc::tma_load_3d(smem + L::OFF_V + c * 8192, &map_v, c * 64, kt.n2, (int)kt.key0,
                                            &bars[F_KV_FULL]);
                }
            }
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i % kQStages, use = tc_i / kQStages;
                const int nt = min(tpt, kt.ntok - i * tpt);
                // this lane's tokens: gather rows 4 lane .. 4 lane + 3 (rows past
                // the last token re-read the first token's row, their P is 0),
                // else tokens lane, lane + 32, ...
                int ent[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tk = gather ? (4 * lane + j) / G : lane + 32 * j;
                    ent[j] = tk < nt ? ws.entries[kt.e0 + i * tpt + tk] : (gather ? ws.entries[kt.e0 + i * tpt] : -1);
                }
                if (use > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(&bars[F_Q_EMPTY + s], (use - 1) & 1, abort_flag,
                                                                       kWaitNs))) {
                    ok = false;
                    break;
                }
                if (lead) {
                    int *m = meta + (tc_i % kMetaF) * kRows;
                    for (int tt = lane; tt < tpt; tt += 32) m[tt] = tt < nt ? ws.entries[kt.e0 + i * tpt + tt] : -1;
                    __syncwarp();
                }
                ++armed_q[s];
                if (lane == 0)
                    tc::mbar_arrive_expect_tx(&bars[F_Q_FULL + s], (uint32_t)my_planes * tpt * G * 128);
                __syncwarp();
                uint8_t *qdst = smem + L::OFF_Q + s * L::Q_STAGE;
                if (gather) {
                    // G in {1, 2, 4}: lane k fetches tile rows 4k..4k+3 with one gather4 per plane
                    int y[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = 4 * lane + j;
                        y[j] = (ent[j] / g.block_count) * g.n1 + kt.n2 * G + row % G;
                    }
                    for (int c = lq; c < KC; c += 2)
                        tc::tma_gather4(qdst + c * 16384 + lane * 512, qmap(c), cx(c), y[0], y[1], y[2], y[3],
                                        &bars[F_Q_FULL + s]);
                } else {
                    // one (token, plane) box per load, tokens over the lanes
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int tt = lane + 32 * j;
                        if (tt >= tpt) break;
                        const int y = ent[j] >= 0 ? (ent[j] / g.block_count) * g.n1 + kt.n2 * G : oob_row;
                        for (int c = lq; c < KC; c += 2)
                            tc::tma_load_2d(qdst + c * 16384 + tt * G * 128, qmap(c), cx(c), y, &bars[F_Q_FULL + s]);
                    }
                }
            }
            ++ne;
        }
        if (!ok && lane == 0) fail();
        // let every load this warp issued land before the CTA exits
        bool drained = tc::drain_armed(&bars[F_KV_FULL], armed_kv, kWaitNs);
        for (int i = 0; i < kQStages; ++i) drained = tc::drain_armed(&bars[F_Q_FULL + i], armed_q[i], kWaitNs) && drained;
        if (!drained && lane == 0) fail();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule; one elected lane issues each
        // instruction.
        const bool bf16 = !kFp16;
        const uint32_t id_s = tc::idesc_f16(kRows, nk, bf16, false, false);
        const uint32_t id_o = tc::idesc_f16(kRows, DV, bf16, false, true);
        const uint32_t ks = sbase + L::OFF_K, vs = sbase + L::OFF_V, ps = sbase + L::OFF_P;
        auto wait = [&](int b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, tc::mbar_wait(&bars[b], parity, abort_flag, kWaitNs));
        };
        int ne = 0, tc_i = 0;
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            if (!wait(F_KV_FULL, ne & 1)) { ok = false; break; }
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i % kQStages, use = tc_i / kQStages;
                if (!wait(F_Q_FULL + s, use & 1)) { ok = false; break; }
                tc::tc_fence_after();
                const uint32_t qs = sbase + L::OFF_Q + s * L::Q_STAGE;
                // S = Q K^T (both operands K-major)
                for (int kk = 0; kk < DQK / 16; ++kk)
                    tc::mma_f16_ss_warp(tmem + kColS, tc::sw128_desc(qs + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                                        tc::sw128_desc(ks + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
                tc::mma_commit_warp(&bars[F_S_FULL]);
                // the softmax is done with S (and its tile's metadata)
                if (!wait(F_P_FULL, tc_i & 1)) { ok = false; break; }
                tc::tc_fence_after();
                tc::mma_commit_warp(&bars[F_Q_EMPTY + s]);
                if (PASS == 2) {
                    // O = P V (A: P K-major, B: V tile MN-major, N = Dv)
                    if (tc_i > 0 && !wait(F_O_FREE, (tc_i - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    for (int kk = 0; kk < nk / 16; ++kk)
                        tc::mma_f16_ss_warp(tmem + kColO, tc::sw128_desc(ps + kk * 32, 16, 1024),
                                            tc::sw128_desc(vs + kk * 2048, 8192, 1024), id_o, kk > 0);
                    tc::mma_commit_warp(&bars[F_O_DONE]);
                }
            }
            if (!ok) break;
            tc::mma_commit_warp(&bars[F_KV_EMPTY]);
            ++ne;
        }
        if (!ok && lane == 0) fail();
        // every MMA issued must be complete before TMEM is freed
        tc::mma_commit_warp(&bars[F_DRAIN]);
        if (!__all_sync(0xffffffffu, tc::mbar_wait_drain(&bars[F_DRAIN], 0, kWaitNs)) && lane == 0) fail();
    } else if (warp < 6) {
        // ------------------------------------------------------ softmax
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                      // query row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const int tt = r / G, gg = r % G;
        uint8_t *prow = smem + L::OFF_P;
        int tc_i = 0;
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                const int s = tc_i % kQStages, use = tc_i / kQStages;
                ok = tc::mbar_wait(&bars[F_Q_FULL + s], use & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const int ent = tt < tpt ? meta[(tc_i % kMetaF) * kRows + tt] : -1;
                const bool valid = ent >= 0;
                const int64_t grow = valid ? (int64_t)(ent / g.block_count) * g.n1 + kt.n2 * G + gg : 0;
                float m2 = 0.f;
                if (PASS == 2 && valid) m2 = mrow[grow] * 1.4426950408889634f;
                ok = tc::mbar_wait(&bars[F_S_FULL], tc_i & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                if (PASS == 1) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c < nk / 16) {
                            uint32_t sv[16];
                            tc::tmem_ld16(trow + kColS + c * 16, sv);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 16; ++j) mx = fmaxf(mx, __uint_as_float(sv[j]) * g.scale);
                        }
                    }
                    tc::tc_fence_before();
                    tc::mbar_arrive(&bars[F_P_FULL]);
                    if (valid) atomic_max_f32(mrow + grow, mx);
                } else {
                    float sum = 0.f;
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c < nk / 16) {
                            uint32_t sv[16];
                            tc::tmem_ld16(trow + kColS + c * 16, sv);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 16; j += 2) {
                                float p0 = 0.f, p1 = 0.f;
                                if (valid) {
                                    p0 = ex2(fmaf(__uint_as_float(sv[j]), g.scale_log2, -m2));
                                    p1 = ex2(fmaf(__uint_as_float(sv[j + 1]), g.scale_log2, -m2));
                                }
                                sum += p0 + p1;
                                pk[c * 8 + j / 2] = pack2<kFp16>(p0, p1);
                            }
                        }
                    }
                    // the previous tile's P V must be done with the P buffer
                    if (tc_i > 0) {
                        ok = tc::mbar_wait(&bars[F_O_DONE], (tc_i - 1) & 1, abort_flag, kWaitNs);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        if (c < nk / 8)
                            *reinterpret_cast<uint4 *>(prow + sw_off(r, c)) =
                                make_uint4(pk[c * 4], pk[c * 4 + 1], pk[c * 4 + 2], pk[c * 4 + 3]);
                    tc::fence_proxy_async_smem();
                    tc::tc_fence_before();
                    tc::mbar_arrive(&bars[F_P_FULL]);
                    if (valid) atomicAdd(lrow + grow, sum);
                }
            }
        }
        if (!ok) fail();
    } else if (PASS == 2) {
        // ------------------------------------------------------ O drain
        const int q4 = warp & 3;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const int tt = (q4 * 32 + lane) / G, gg = (q4 * 32 + lane) % G;
        uint8_t *stg = smem + L::OFF_STG + (warp - 6) * 4096;
        int tc_i = 0;
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < g.n_units && ok; ti += gridDim.x) {
            const KeyTile kt = decode(g, ws, ti, nk, tpt);
            if (kt.ntok == 0) continue;
            for (int i = 0; i < kt.ntiles; ++i, ++tc_i) {
                ok = tc::mbar_wait(&bars[F_O_DONE], tc_i & 1, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::tc_fence_after();
                const int ent = tt < tpt ? meta[(tc_i % kMetaF) * kRows + tt] : -1;
                const int64_t grow = ent >= 0 ? (int64_t)(ent / g.block_count) * g.n1 + kt.n2 * G + gg : -1;
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t v0[16], v1[16];
                    tc::tmem_ld16(trow + kColO + c * 32, v0);
                    tc::tmem_ld16(trow + kColO + c * 32 + 16, v1);
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
                        if (gr >= 0) tc::red_add_v4(oacc + gr * DV + c * 32 + j4 * 4, x.x, x.y, x.z, x.w);
                    }
                    __syncwarp();
                }
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[F_O_FREE]);
            }
        }
        if (!ok) fail();
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 256);
    }
}

// m = -inf, l = 0, O_acc = 0 for every query row
__global__ void k_fwd_init(float *__restrict__ mrow, float *__restrict__ lrow, float4 *__restrict__ oacc,
                           int64_t rows) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * 32; i += stride) {
        oacc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < rows) {
            mrow[i] = -INFINITY;
            lrow[i] = 0.f;
        }
    }
}

// one warp per query row: O = O_acc / l (rounded to the dtype), stats x 8
template <bool kFp16>
__global__ void k_fwd_finalize(const float *__restrict__ mrow, const float *__restrict__ lrow,
                               const float4 *__restrict__ oacc, uint2 *__restrict__ o, float *__restrict__ smax,
                               float *__restrict__ ssum, int64_t rows) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nw) {
        // every valid row has l >= 1 (its maximum term is exp(0)); l == 0 marks a
        // row that selected nothing (BSND padding): zeros in all outputs
        const float l = lrow[r], inv = l > 0.f ? 1.f / l : 0.f;
        const float4 a = oacc[r * 32 + lane];
        o[r * 32 + lane] = make_uint2(pack2<kFp16>(a.x * inv, a.y * inv), pack2<kFp16>(a.z * inv, a.w * inv));
        if (lane < 8) smax[r * 8 + lane] = l > 0.f ? mrow[r] : 0.f;
        else if (lane < 16) ssum[r * 8 + lane - 8] = l;
    }
}

template <bool kFp16, int DQK, int PASS>
cudaError_t launch_fwd_t(const Geometry &g, const Workspace &ws, const sag_io &io, cudaStream_t s, int num_sms) {
    FwdArgs a;
    a.g = g;
    a.ws = ws;
    a.nk = g.block_size > 64 ? 64 : g.block_size;
    a.tpt = kRows / g.group;
    QkMaps m;
    CUtensorMap mv;
    const uint32_t box_rows = (g.group <= 4 && 4 % g.group == 0) ? 1 : g.group;
    if (!qk_maps(&m, g, io, kFp16, box_rows, a.nk) || !tmap_3d(&mv, io.value, kFp16, 128, g.n2, g.t2, a.nk))
        return cudaErrorInvalidValue;
    auto fn = k_fwd_tc<kFp16, DQK, PASS>;
    const int smem = FwdSmem<DQK>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int64_t grid = g.n_units < num_sms ? g.n_units : num_sms;
    if (grid < 1) grid = 1;
    fn<<<(int)grid, kFwdThreads, smem, s>>>(m.q, m.k, mv, m.qr, m.kr, a);
    return cudaGetLastError();
}

template <bool kFp16, int PASS>
cudaError_t launch_fwd_d(const Geometry &g, const Workspace &ws, const sag_io &io, cudaStream_t s, int num_sms) {
    return g.d_qk == 192 ? launch_fwd_t<kFp16, 192, PASS>(g, ws, io, s, num_sms)
                         : launch_fwd_t<kFp16, 128, PASS>(g, ws, io, s, num_sms);
}

}  // namespace

bool fwd_tc_supported(const Geometry &g) { return bwd_tc_supported(g); }

cudaError_t launch_fwd_init(const Geometry &g, const Workspace &ws, cudaStream_t s, int num_sms) {
    const int64_t rows = (int64_t)g.t1 * g.n1;
    int64_t blocks = (rows * 32 + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    if (blocks < 1) blocks = 1;
    k_fwd_init<<<(int)blocks, 256, 0, s>>>(ws.lse2, ws.delta, reinterpret_cast<float4 *>(ws.dq_acc), rows);
    return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const Geometry &g, const Workspace &ws, const sag_io &io, int pass, bool fp16,
                          cudaStream_t s, int num_sms) {
    if (!fwd_tc_supported(g) || (pass != 1 && pass != 2)) return cudaErrorInvalidValue;
    if (fp16) return pass == 1 ? launch_fwd_d<true, 1>(g, ws, io, s, num_sms) : launch_fwd_d<true, 2>(g, ws, io, s, num_sms);
    return pass == 1 ? launch_fwd_d<false, 1>(g, ws, io, s, num_sms) : launch_fwd_d<false, 2>(g, ws, io, s, num_sms);
}

cudaError_t launch_fwd_finalize(const Geometry &g, const Workspace &ws, void *o, float *smax, float *ssum, bool fp16,
                                cudaStream_t s, int num_sms) {
    const int64_t rows = (int64_t)g.t1 * g.n1;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    if (blocks < 1) blocks = 1;
    const float4 *acc = reinterpret_cast<const float4 *>(ws.dq_acc);
    if (fp16)
        k_fwd_finalize<true><<<(int)blocks, 256, 0, s>>>(ws.lse2, ws.delta, acc, static_cast<uint2 *>(o), smax, ssum,
                                                        rows);
    else
        k_fwd_finalize<false><<<(int)blocks, 256, 0, s>>>(ws.lse2, ws.delta, acc, static_cast<uint2 *>(o), smax,
                                                         ssum, rows);
    return cudaGetLastError();
}

}  // namespace sag
