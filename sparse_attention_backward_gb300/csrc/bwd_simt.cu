// CUDA-core (SIMT) key-block-major backward.
//
// One CTA per item (batch, KV head, key block).  The block's bs key and value
// rows stay in shared memory as fp32; warp w owns keys [8w, 8w+8) and keeps
// their dK / dV accumulators in registers for the whole bucket, so dK and dV
// need no atomics and are reduced in bucket (token) order.  For every query
// row (token from the bucket, head g of the group):
//   s_j  = <q, k_j>,  P_j = exp2(s_j * scale*log2e - lse2)
//   dP_j = <dY, v_j>, dS_j = P_j (dP_j - Delta)
//   dV_j += P_j dY,   dK_j += dS_j q   (scale applied once at the end)
//   dQ   += dS_j k_j  (fp32 atomics, or dS stored for the fixed-order pass)
// ("NsaSelectedAttentionGrad" README, function description; softmax adjoint
// of "aclnnFlashAttentionUnpaddingScoreGradV3", Formula.)
#include "kernels.cuh"

namespace sag {

constexpr int kKeysPerWarp = 8;
constexpr int kRowsPerStep = 8;

template <bool kFp16, int DQK, int DV>
__global__ void __launch_bounds__(512) k_bwd_simt(Geometry g, Workspace ws,
                                                  const uint16_t *__restrict__ q,
                                                  const uint16_t *__restrict__ k,
                                                  const uint16_t *__restrict__ v,
                                                  const uint16_t *__restrict__ dy,
                                                  uint16_t *__restrict__ dk,
                                                  uint16_t *__restrict__ dv, int deterministic) {
    constexpr int MQ = DQK / 32, MV = DV / 32;
    extern __shared__ float smem[];
    const int bs = g.block_size;
    float *sk = smem;                                 // [bs][DQK]
    float *sv = sk + bs * DQK;                        // [bs][DV]
    float *sq = sv + bs * DV;                         // [R][DQK]
    float *sy = sq + kRowsPerStep * DQK;              // [R][DV]
    float *slse = sy + kRowsPerStep * DV;             // [R]
    float *sdel = slse + kRowsPerStep;                // [R]
    int *smeta = reinterpret_cast<int *>(sdel + kRowsPerStep);  // [R] (t*N1+h) or -1
    int *sslot = smeta + kRowsPerStep;                // [R] slot*G + g (dS store)

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j0 = warp * kKeysPerWarp;

    for (int64_t item = blockIdx.x; item < g.n_items; item += gridDim.x) {
        const int b = batch_of_item(ws.item_base, g.batch, item);
        const int nblk = (ws.cu_kv[b + 1] - ws.cu_kv[b]) / bs;
        const int64_t local = item - ws.item_base[b];
        const int n2 = (int)(local / nblk);
        const int kb = (int)(local % nblk);
        const int64_t key0 = ws.cu_kv[b] + (int64_t)kb * bs;   // first key row of the block

        __syncthreads();
        for (int i = threadIdx.x; i < bs * DQK; i += blockDim.x) {
            const int r = i / DQK, d = i % DQK;
            sk[i] = u16_to_f<kFp16>(k[((key0 + r) * g.n2 + n2) * DQK + d]);
        }
        for (int i = threadIdx.x; i < bs * DV; i += blockDim.x) {
            const int r = i / DV, d = i % DV;
            sv[i] = u16_to_f<kFp16>(v[((key0 + r) * g.n2 + n2) * DV + d]);
        }

        float acc_k[kKeysPerWarp][MQ], acc_v[kKeysPerWarp][MV];
#pragma unroll
        for (int j = 0; j < kKeysPerWarp; ++j) {
#pragma unroll
            for (int m = 0; m < MQ; ++m) acc_k[j][m] = 0.f;
#pragma unroll
            for (int m = 0; m < MV; ++m) acc_v[j][m] = 0.f;
        }

        // the bucket is sorted by token: take the entries of this launch's chunk
        const int e_end = ws.offset[item + 1];
        const int e0 = lower_bound_token(ws.entries, ws.offset[item], e_end, g.tok_lo, g.block_count);
        const int e1 = lower_bound_token(ws.entries, e0, e_end, g.tok_hi, g.block_count);
        const int64_t nrows = (int64_t)(e1 - e0) * g.group;
        for (int64_t r0 = 0; r0 < nrows; r0 += kRowsPerStep) {
            __syncthreads();
            // stage up to R query rows (entry = r / G, head g = r % G)
            for (int i = threadIdx.x; i < kRowsPerStep * (DQK + DV); i += blockDim.x) {
                const int rr = i / (DQK + DV), d = i % (DQK + DV);
                const int64_t r = r0 + rr;
                float x = 0.f;
                if (r < nrows) {
                    const int ent = ws.entries[e0 + r / g.group];
                    const int t = ent / g.block_count;
                    const int h = n2 * g.group + (int)(r % g.group);
                    const int64_t row = (int64_t)t * g.n1 + h;
                    x = d < DQK ? u16_to_f<kFp16>(q[row * DQK + d]) : u16_to_f<kFp16>(dy[row * DV + d - DQK]);
                }
                if (d < DQK) sq[rr * DQK + d] = x; else sy[rr * DV + d - DQK] = x;
            }
            if (threadIdx.x < kRowsPerStep) {
                const int64_t r = r0 + threadIdx.x;
                if (r < nrows) {
                    const int ent = ws.entries[e0 + r / g.group];
                    const int t = ent / g.block_count, slot = ent % g.block_count;
                    const int gg = (int)(r % g.group);
                    const int64_t row = (int64_t)t * g.n1 + n2 * g.group + gg;
                    smeta[threadIdx.x] = (int)row;
                    sslot[threadIdx.x] = slot * g.group + gg;
                    slse[threadIdx.x] = ws.lse2[row];
                    sdel[threadIdx.x] = ws.delta[row];
                } else {
                    smeta[threadIdx.x] = -1;
                }
            }
            __syncthreads();
            for (int rr = 0; rr < kRowsPerStep; ++rr) {
                const int row = smeta[rr];
                if (row < 0) break;
                float qv[MQ], yv[MV], dq[MQ];
#pragma unroll
                for (int m = 0; m < MQ; ++m) { qv[m] = sq[rr * DQK + lane + 32 * m]; dq[m] = 0.f; }
#pragma unroll
                for (int m = 0; m < MV; ++m) yv[m] = sy[rr * DV + lane + 32 * m];
                const float lse2 = slse[rr], del = sdel[rr];
                float ds_mine = 0.f;
#pragma unroll
                for (int j = 0; j < kKeysPerWarp; ++j) {
                    const float *kr = sk + (j0 + j) * DQK;
                    const float *vr = sv + (j0 + j) * DV;
                    float s = 0.f, dp = 0.f;
#pragma unroll
                    for (int m = 0; m < MQ; ++m) s = fmaf(qv[m], kr[lane + 32 * m], s);
#pragma unroll
                    for (int m = 0; m < MV; ++m) dp = fmaf(yv[m], vr[lane + 32 * m], dp);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        s += __shfl_xor_sync(0xffffffffu, s, o);
                        dp += __shfl_xor_sync(0xffffffffu, dp, o);
                    }
                    const float p = exp2f(fmaf(s, g.scale_log2, -lse2));
                    const float ds = p * (dp - del);
                    if (lane == j) ds_mine = ds;
#pragma unroll
                    for (int m = 0; m < MV; ++m) acc_v[j][m] = fmaf(p, yv[m], acc_v[j][m]);
#pragma unroll
                    for (int m = 0; m < MQ; ++m) {
                        acc_k[j][m] = fmaf(ds, qv[m], acc_k[j][m]);
                        dq[m] = fmaf(ds, kr[lane + 32 * m], dq[m]);
                    }
                }
                if (deterministic) {
                    // dS[t][n2][slot][g][j] in the input dtype
                    if (lane < kKeysPerWarp) {
                        const int t = row / g.n1 - g.tok_lo;
                        const int64_t base = (((int64_t)t * g.n2 + n2) * g.block_count * g.group + sslot[rr]) * bs;
                        ws.ds[base + j0 + lane] = f_to_u16<kFp16>(ds_mine);
                    }
                } else {
                    float *dst = ws.dq_acc + (int64_t)row * DQK;
#pragma unroll
                    for (int m = 0; m < MQ; ++m) atomicAdd(dst + lane + 32 * m, dq[m]);
                }
            }
        }
        // write dK = scale * acc_k and dV = acc_v for this warp's keys, or
        // carry them in fp32 (dK unscaled) when the tokens come in chunks
#pragma unroll
        for (int j = 0; j < kKeysPerWarp; ++j) {
            const int64_t row = (key0 + j0 + j) * g.n2 + n2;
            if (g.chunked) {
                float *acc = ws.dkv_acc + row * (DQK + DV);
#pragma unroll
                for (int m = 0; m < MQ; ++m) acc[lane + 32 * m] += acc_k[j][m];
#pragma unroll
                for (int m = 0; m < MV; ++m) acc[DQK + lane + 32 * m] += acc_v[j][m];
            } else {
#pragma unroll
                for (int m = 0; m < MQ; ++m) dk[row * DQK + lane + 32 * m] = f_to_u16<kFp16>(acc_k[j][m] * g.scale);
#pragma unroll
                for (int m = 0; m < MV; ++m) dv[row * DV + lane + 32 * m] = f_to_u16<kFp16>(acc_v[j][m]);
            }
        }
    }
}

// dQ[t, n2*G+g] = scale * sum_slot sum_r dS[t][n2][slot][g][r] * K[row(slot, r)]
// in slot order then key order: one CTA per (t, n2).
// Fixed-order dQ from the stored dS on CUDA cores (deterministic mode, for
// shapes the tensor-core pass does not take):
//     dQ[t, h] = scale * sum over slots in list order, keys in block order, of
//                dS[t, h, slot, key] * K[key row]
// One warp per (token, KV head) and group of up to HPW query heads (HPW = 1,
// 2, 4 or 8, the smallest that covers G up to 8: fewer accumulators, more
// warps and loads in flight); lane l owns head dims [l * DQK/32,
// (l + 1) * DQK/32) of those heads.  No shared memory and no block barrier: a
// key row is one coalesced warp load, the dS value of a head a broadcast load.
template <bool kFp16, int DQK, int kHeadsPerWarp>
__global__ void __launch_bounds__(256) k_dq_from_ds(Geometry g, Workspace ws,
                                                    const uint16_t *__restrict__ k,
                                                    const uint16_t *__restrict__ k_rope,
                                                    const int32_t *__restrict__ topk,
                                                    uint16_t *__restrict__ dq, uint16_t *__restrict__ dq_rope) {
    constexpr int DPL = DQK / 32;                       // dims per lane: 4 or 6
    const int bs = g.block_size, G = g.group;
    const int d_main = DQK - g.d_rope;
    const int lane = threadIdx.x & 31;
    const int hgroups = (G + kHeadsPerWarp - 1) / kHeadsPerWarp;
    const int64_t nwork = (int64_t)(g.tok_hi - g.tok_lo) * g.n2 * hgroups;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t wk = (((int64_t)blockIdx.x * blockDim.x) >> 5) + (threadIdx.x >> 5); wk < nwork; wk += warps) {
        const int64_t cp = wk / hgroups;                // pair index inside the chunk
        const int h0 = (int)(wk % hgroups) * kHeadsPerWarp;
        const int nh = min(kHeadsPerWarp, G - h0);
        const int t = g.tok_lo + (int)(cp / g.n2), n2 = (int)(cp % g.n2);
        const int64_t pair = (int64_t)t * g.n2 + n2;
        const int b = batch_of(ws.cu_q, g.batch, t);
        const int nblk = t < ws.q_end[b] ? ws.kv_blocks[b] : 0;   // ids must be below; none for padding
        float acc[kHeadsPerWarp][DPL];
#pragma unroll
        for (int h = 0; h < kHeadsPerWarp; ++h)
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
        for (int slot = 0; slot < g.block_count; ++slot) {
            const int id = __ldg(topk + pair * g.block_count + slot);
            if (id < 0 || id >= nblk) continue;       // reported by the histogram
            const int64_t key0 = ws.cu_kv[b] + (int64_t)id * bs;
            const uint16_t *dsrow = ws.ds + ((cp * g.block_count + slot) * (int64_t)G + h0) * bs;
#pragma unroll 4
            for (int r = 0; r < bs; ++r) {
                const int64_t krow = (key0 + r) * g.n2 + n2;
                // the lane's DPL dims in pairs (4-byte loads; a pair never
                // straddles the rope boundary: both offsets are even)
                float kv[DPL];
#pragma unroll
                for (int e = 0; e < DPL; e += 2) {
                    const int d = lane * DPL + e;
                    const uint32_t two = d < d_main ? __ldg(reinterpret_cast<const uint32_t *>(k + krow * d_main + d))
                                                    : __ldg(reinterpret_cast<const uint32_t *>(
                                                          k_rope + krow * g.d_rope + d - d_main));
                    kv[e] = u16_to_f<kFp16>((uint16_t)(two & 0xffffu));
                    kv[e + 1] = u16_to_f<kFp16>((uint16_t)(two >> 16));
                }
#pragma unroll
                for (int h = 0; h < kHeadsPerWarp; ++h) {
                    if (h >= nh) break;
                    const float sv = u16_to_f<kFp16>(dsrow[(int64_t)h * bs + r]);
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(sv, kv[e], acc[h][e]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < kHeadsPerWarp; ++h) {
            if (h >= nh) break;
            const int64_t row = (int64_t)t * g.n1 + (int64_t)n2 * G + h0 + h;
#pragma unroll
            for (int e = 0; e < DPL; ++e)
                *split_col(dq, dq_rope, row, lane * DPL + e, DQK, g.d_rope) = f_to_u16<kFp16>(acc[h][e] * g.scale);
        }
    }
}

// dK = scale * acc[:, :d_qk], dV = acc[:, d_qk:] after the last chunk.
template <bool kFp16>
__global__ void __launch_bounds__(256) k_cast_dkv(Geometry g, const float *__restrict__ acc,
                                                  uint16_t *__restrict__ dk, uint16_t *__restrict__ dk_rope,
                                                  uint16_t *__restrict__ dv) {
    const int w = g.d_qk + g.d_v;
    const int64_t n = (int64_t)g.t2 * g.n2 * w;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / w;
        const int c = (int)(i % w);
        if (c < g.d_qk) *split_col(dk, dk_rope, row, c, g.d_qk, g.d_rope) = f_to_u16<kFp16>(acc[i] * g.scale);
        else dv[row * g.d_v + c - g.d_qk] = f_to_u16<kFp16>(acc[i]);
    }
}

cudaError_t launch_cast_dkv(const Geometry &g, const Workspace &ws, void *dk, void *dk_rope, void *dv, bool fp16,
                            cudaStream_t s, int num_sms) {
    const int64_t n = (int64_t)g.t2 * g.n2 * (g.d_qk + g.d_v);
    int64_t grid = (n + 255) / 256;
    if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
    if (fp16)
        k_cast_dkv<true><<<(int)grid, 256, 0, s>>>(g, ws.dkv_acc, (uint16_t *)dk, (uint16_t *)dk_rope, (uint16_t *)dv);
    else
        k_cast_dkv<false><<<(int)grid, 256, 0, s>>>(g, ws.dkv_acc, (uint16_t *)dk, (uint16_t *)dk_rope,
                                                    (uint16_t *)dv);
    return cudaGetLastError();
}

template <bool kFp16, int DQK, int DV>
static cudaError_t launch_simt_t(const Geometry &g, const Workspace &ws, const sag_io &io, bool det, cudaStream_t s,
                                 int num_sms) {
    const int threads = (g.block_size / kKeysPerWarp) * 32;
    const size_t smem = sizeof(float) * ((size_t)g.block_size * (DQK + DV) + kRowsPerStep * (DQK + DV) +
                                         2 * kRowsPerStep) + 2 * sizeof(int) * kRowsPerStep;
    auto fn = k_bwd_simt<kFp16, DQK, DV>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int64_t grid = g.n_items;
    if (grid > (int64_t)num_sms * 64) grid = (int64_t)num_sms * 64;
    fn<<<(int)grid, threads, smem, s>>>(g, ws, (const uint16_t *)io.query, (const uint16_t *)io.key,
                                        (const uint16_t *)io.value, (const uint16_t *)io.attention_out_grad,
                                        (uint16_t *)io.dk, (uint16_t *)io.dv, det ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, bool deterministic,
                            cudaStream_t s, int num_sms) {
    if (g.d_rope) return cudaErrorInvalidValue;   // the rope split runs on the tensor-core kernels only
#define SAG_SIMT_CASE(F, A, B) \
    if (fp16 == F && g.d_qk == A && g.d_v == B) return launch_simt_t<F, A, B>(g, ws, io, deterministic, s, num_sms);
    SAG_SIMT_CASE(false, 192, 128) SAG_SIMT_CASE(false, 128, 128) SAG_SIMT_CASE(false, 192, 192)
    SAG_SIMT_CASE(false, 128, 192) SAG_SIMT_CASE(true, 192, 128) SAG_SIMT_CASE(true, 128, 128)
    SAG_SIMT_CASE(true, 192, 192) SAG_SIMT_CASE(true, 128, 192)
#undef SAG_SIMT_CASE
    return cudaErrorInvalidValue;
}

template <bool kFp16, int DQK, int HPW>
static cudaError_t launch_dq_h(const Geometry &g, const Workspace &ws, const sag_io &io, cudaStream_t s,
                               int num_sms) {
    const int hgroups = (g.group + HPW - 1) / HPW;
    const int64_t warps = (int64_t)(g.tok_hi - g.tok_lo) * g.n2 * hgroups;
    int64_t grid = (warps + 7) / 8;
    if (grid > (int64_t)num_sms * 32) grid = (int64_t)num_sms * 32;
    if (grid == 0) return cudaSuccess;
    k_dq_from_ds<kFp16, DQK, HPW><<<(int)grid, 256, 0, s>>>(g, ws, (const uint16_t *)io.key,
                                                            (const uint16_t *)io.key_rope, io.topk_indices,
                                                            (uint16_t *)io.dq, (uint16_t *)io.dq_rope);
    return cudaGetLastError();
}

template <bool kFp16, int DQK>
static cudaError_t launch_dq_t(const Geometry &g, const Workspace &ws, const sag_io &io, cudaStream_t s,
                               int num_sms) {
    if (g.group == 1) return launch_dq_h<kFp16, DQK, 1>(g, ws, io, s, num_sms);
    if (g.group == 2) return launch_dq_h<kFp16, DQK, 2>(g, ws, io, s, num_sms);
    if (g.group <= 4) return launch_dq_h<kFp16, DQK, 4>(g, ws, io, s, num_sms);
    return launch_dq_h<kFp16, DQK, 8>(g, ws, io, s, num_sms);
}

cudaError_t launch_dq_from_ds(const Geometry &g, const Workspace &ws, const sag_io &io, bool fp16, cudaStream_t s,
                              int num_sms) {
    if (fp16) return g.d_qk == 192 ? launch_dq_t<true, 192>(g, ws, io, s, num_sms) : launch_dq_t<true, 128>(g, ws, io, s, num_sms);
    return g.d_qk == 192 ? launch_dq_t<false, 192>(g, ws, io, s, num_sms) : launch_dq_t<false, 128>(g, ws, io, s, num_sms);
}

}  // namespace sag
