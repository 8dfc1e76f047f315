/*
 * selattn.h -- C ABI of the GB300 selected-attention backward library
 * (libselattn.so).
 *
 * The operation is the training backward of NSA-style selected attention as
 * the "NsaSelectedAttentionGrad" README (ops-transformer) defines it:
 *
 *   function description: for every query token and KV head, gather
 *     selectedBlockCount blocks of selectedBlockSize key / value rows named by
 *     topkIndices (selectedKey = Gather(key, topkIndices[i])), then run the
 *     attention backward over the gathered rows:
 *         dV = P^T dY,   dQ = dS K / sqrt(d),   dK = dS^T Q / sqrt(d)
 *     with dK and dV scatter-added back to the gathered key rows;
 *   parameters: query, key, value, attentionOut, attentionOutGrad (bf16 or
 *     fp16), softmaxMax and softmaxSum (fp32 forward intermediates),
 *     topkIndices (int32), scaleValue (double, the 1/sqrt(d) of the formula);
 *     outputs dqOut, dkOut, dvOut in the input dtype;
 *   constraints: TND layout, N1 a multiple of N2 with G = N1/N2 in [1, 32],
 *     D in {128, 192}, block size a multiple of 16 and <= 128, block count in
 *     [1, 128], count * size < 8192, per-batch S2 a multiple of the block size
 *     and at least count * size, stats [T1, N1, 8], topkIndices
 *     [T1, N2, selectedBlockCount].
 *
 * With P = exp(scale * Q K_sel^T - lse), lse = softmaxMax + ln(softmaxSum)
 * (lane 0 of the 8), Delta = rowsum(dY * O) and dS = P * (dY V_sel^T - Delta)
 * (the softmax adjoint behind the dense formulas of the
 * "aclnnFlashAttentionUnpaddingScoreGradV3" page).
 *
 * The calling convention is the two-phase one those pages describe: phase 1
 * validates the parameters and returns the workspace size; phase 2 takes the
 * caller's workspace and a stream and enqueues the work.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, 16-byte aligned, densely packed
 *     in TND order (row-major, last dimension contiguous).  cu_seqlens_* in
 *     the descriptor are HOST arrays.
 *   - The caller owns every buffer, including the workspace.  The library
 *     allocates no memory and keeps no state between calls.
 *   - Inputs are never written.  dq, dk and dv are fully overwritten; key rows
 *     that no query selected get dK = dV = 0.
 *   - Host-side problems are reported synchronously, before anything is
 *     enqueued.  Problems found by the device (a block id out of range, a
 *     bounded wait that ran out) are recorded in the workspace and read back
 *     with sel_attn_grad_query_error.
 *   - An entry point that takes a stream makes the device owning that stream
 *     current for the length of the call and gives the calling thread its
 *     previous current device back before returning.
 */
#ifndef SELATTN_H
#define SELATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sag_status {
    SAG_OK = 0,
    SAG_ERR_NULL = 1,        /* a required pointer (or the descriptor) is NULL */
    SAG_ERR_SHAPE = 2,       /* a size or length outside the constraints */
    SAG_ERR_DTYPE = 3,       /* dtype is neither SAG_BF16 nor SAG_FP16 */
    SAG_ERR_UNSUPPORTED = 4, /* allowed by the constraints but not built here */
    SAG_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than phase 1 said */
    SAG_ERR_ALIGN = 6,       /* a device pointer is not 16-byte aligned */
    SAG_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
    SAG_ERR_INDEX = 8,       /* device: a topkIndices entry outside [0, S2_b / block_size) */
    SAG_ERR_TIMEOUT = 9      /* device: a bounded wait in a kernel ran out */
} sag_status;

typedef enum sag_dtype { SAG_BF16 = 0, SAG_FP16 = 1 } sag_dtype;

/*
 * Problem descriptor.
 *   batch          B >= 1
 *   cu_seqlens_q   host int32[B+1]: prefix sums of the query lengths, [0] = 0.
 *                  A batch may have no query tokens.  In TND the last entry
 *                  is T1; in BSND these are the valid lengths of the padded
 *                  rows (see layout).
 *   cu_seqlens_kv  host int32[B+1]: prefix sums of the key lengths; every
 *                  batch's S2 is a multiple of block_size and >= block_size *
 *                  block_count.
 *   n1, n2         query heads and key/value heads (N1 % N2 == 0, N1/N2 <= 32)
 *   d_qk, d_v      head dims of query/key and of value/attentionOut/dY
 *                  (each 128 or 192; with d_rope, d_qk is the non-rope part
 *                  and must be 128)
 *   block_size     selectedBlockSize (multiple of 16, <= 128)
 *   block_count    selectedBlockCount (1..128, block_size * block_count < 8192)
 *   dtype          sag_dtype of every 16-bit tensor
 *   deterministic  0: default mode (dQ reduced with fp32 atomics, results may
 *                  differ in the last bits between runs); 1: every output is
 *                  bit-identical run to run
 *   layout         SAG_LAYOUT_TND (0): tokens of all batches packed, rows
 *                  cu_seqlens[b] .. cu_seqlens[b+1]-1 belong to batch b.
 *                  SAG_LAYOUT_BSND (1): [B, S, N, D] with every batch padded
 *                  to s1_max query rows and s2_max key rows: token s of batch b
 *                  is row b * s1_max + s (b * s2_max + s for keys); only the
 *                  first S1_b / S2_b rows (from cu_seqlens) are valid.  Padding
 *                  rows are never read for the result (topk_indices rows of
 *                  padding tokens are ignored) and get zero gradients.
 *                  ("aclnnLightningIndexerGrad" page: TND or BSND layouts;
 *                  "NsaSelectedAttentionGrad" README, calling section: a
 *                  non-TND sample.)
 *   scale          scaleValue
 *   s1_max, s2_max BSND only (0 in TND): padded query / key length, <= 128K;
 *                  s2_max a multiple of block_size; B * s1_max and B * s2_max
 *                  <= 2M
 *   d_rope         0, or 64: the query and key head dims are split into a
 *                  d_qk part and a rope part held in separate tensors,
 *                  Q = [query, queryRope], K = [key, keyRope] along D, with
 *                  gradients dq / dqRope and dk / dkRope the matching column
 *                  slices of dQ and dK ("aclnnFlashAttentionUnpaddingScore-
 *                  GradV3" formula section).  Needs the tensor-core path:
 *                  d_qk == 128, d_v == 128.
 */
typedef enum sag_layout { SAG_LAYOUT_TND = 0, SAG_LAYOUT_BSND = 1 } sag_layout;

typedef struct sag_desc {
    int32_t batch;
    int32_t n1, n2;
    int32_t d_qk, d_v;
    int32_t block_size, block_count;
    int32_t dtype;
    int32_t deterministic;
    int32_t layout;
    double scale;
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_kv;
    int32_t s1_max, s2_max;
    int32_t d_rope;
    int32_t reserved_;   /* must be 0 */
} sag_desc;

/*
 * Tensors of one call (device pointers, 16-byte aligned, dense).  Rows are
 * tokens in the descriptor's layout: R1 = T1 (TND) or B * s1_max (BSND),
 * R2 = T2 or B * s2_max.
 *   query               [R1, n1, d_qk]   dtype
 *   key                 [R2, n2, d_qk]   dtype
 *   value               [R2, n2, d_v]    dtype
 *   attention_out       [R1, n1, d_v]    dtype (backward; required: Delta needs it)
 *   attention_out_grad  [R1, n1, d_v]    dtype (backward)
 *   softmax_max         [R1, n1, 8]      fp32 (backward: lane 0 is read; forward: written)
 *   softmax_sum         [R1, n1, 8]      fp32 (idem)
 *   topk_indices        [R1, n2, block_count] int32, block ids local to the
 *                       token's batch
 *   query_rope          [R1, n1, d_rope] dtype, NULL unless d_rope
 *   key_rope            [R2, n2, d_rope] dtype, NULL unless d_rope
 *   dq, dk, dv          like query, key, value: written by the backward
 *   dq_rope, dk_rope    like query_rope, key_rope: written (NULL unless d_rope)
 * The forward writes attention_out, softmax_max and softmax_sum and ignores
 * attention_out_grad and the gradients.
 */
typedef struct sag_io {
    const void *query, *key, *value;
    void *attention_out;              /* read (never written) by the backward, written by the forward */
    const void *attention_out_grad;
    float *softmax_max, *softmax_sum; /* likewise */
    const int32_t *topk_indices;
    const void *query_rope, *key_rope;
    void *dq, *dk, *dv;
    void *dq_rope, *dk_rope;
} sag_io;

/*
 * Phase 1.  Validates the descriptor against the constraints (host only, no
 * CUDA call) and writes the workspace size in bytes the problem needs.
 * Returns SAG_OK, SAG_ERR_NULL, SAG_ERR_SHAPE, SAG_ERR_DTYPE or
 * SAG_ERR_UNSUPPORTED.  SAG_ERR_UNSUPPORTED marks a problem the constraints
 * allow but this library does not take: more than 2^31 - 1 selections in all
 * (T1 * n2 * block_count; the inverted index is 32-bit), or more key blocks
 * in all (sum over batches of n2 * S2_b / block_size) than its scan holds
 * (2^24).
 */
sag_status sel_attn_grad_workspace_size(const sag_desc *desc, size_t *workspace_bytes);

/*
 * Phase 2.  Enqueues the whole backward on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and returns without waiting.
 *   query               [T1, n1, d_qk]   dtype
 *   key                 [T2, n2, d_qk]   dtype
 *   value               [T2, n2, d_v]    dtype
 *   attention_out       [T1, n1, d_v]    dtype (required: Delta needs it)
 *   attention_out_grad  [T1, n1, d_v]    dtype
 *   softmax_max         [T1, n1, 8]      fp32 (lane 0 is read)
 *   softmax_sum         [T1, n1, 8]      fp32 (lane 0 is read)
 *   topk_indices        [T1, n2, block_count] int32, block ids local to the
 *                       token's batch
 *   dq                  [T1, n1, d_qk]   dtype, written
 *   dk                  [T2, n2, d_qk]   dtype, written
 *   dv                  [T2, n2, d_v]    dtype, written
 *   workspace           device scratch of at least the phase-1 size; its
 *                       contents are undefined between calls and two calls in
 *                       flight at once must not share it
 * Returns SAG_OK once enqueued, or a host-side status (nothing enqueued), or
 * SAG_ERR_CUDA when a launch failed.
 */
sag_status sel_attn_grad(const sag_desc *desc, const void *query, const void *key,
                         const void *value, const void *attention_out,
                         const void *attention_out_grad, const float *softmax_max,
                         const float *softmax_sum, const int32_t *topk_indices, void *dq,
                         void *dk, void *dv, void *workspace, size_t workspace_bytes,
                         void *stream);

/*
 * Waits for `stream` and returns the status the device recorded in
 * `workspace` during the last sel_attn_grad on it: SAG_OK, SAG_ERR_INDEX
 * (the offending selections were skipped; outputs are not meaningful) or
 * SAG_ERR_TIMEOUT.  SAG_ERR_CUDA if the wait or the read fails.
 */
sag_status sel_attn_grad_query_error(const void *workspace, void *stream);

/*
 * Phase 2 with every tensor in one sag_io (the form that takes the rope
 * tensors) and two optional cudaEvent_t handles recorded around the main
 * kernel as in sel_attn_grad_timed (NULL = not recorded).  Arguments,
 * ownership and errors are those of sel_attn_grad; SAG_ERR_NULL also when
 * d_rope is set and a rope pointer is NULL.
 */
sag_status sel_attn_grad_ex(const sag_desc *desc, const sag_io *io, void *workspace,
                            size_t workspace_bytes, void *stream, void *main_start, void *main_stop);

/*
 * Launch plan of a problem (host only, no CUDA call): what sel_attn_grad will
 * enqueue for `desc`.
 *   workspace_bytes   same value as sel_attn_grad_workspace_size
 *   launches          kernels one call launches (memsets and copies excluded)
 *   items             key blocks (batch, KV head, block id) the work is split into
 *   token_chunks      query-token chunks the deterministic mode runs in (1 otherwise)
 *   main_kernel       0: CUDA-core kernel, 1: tensor-core (tcgen05) kernel (one of
 *                     two schedules: the softmax between the MMA groups, or, for
 *                     query groups G = n1 / n2 of 1, 2 or 4, split in two phases
 *                     beside them)
 *   dq_path           0: dQ reduced with fp32 atomics inside the main kernel;
 *                     1: dS stored and dQ formed by a fixed-order pass (always
 *                     in deterministic mode; in default mode when it moves
 *                     fewer bytes by the library's count);
 *                     2: the main kernel stores every key tile's fp32 dQ
 *                     partial per (query row, slot) and a pass sums them in
 *                     list order (deterministic mode, when that moves fewer
 *                     bytes than path 1: small blocks and query groups)
 */
typedef struct sag_plan_info {
    uint64_t workspace_bytes;
    int32_t launches;
    int32_t token_chunks;
    int64_t items;
    int32_t main_kernel;
    int32_t dq_path;
} sag_plan_info;

sag_status sel_attn_grad_plan_info(const sag_desc *desc, sag_plan_info *info);

/*
 * sel_attn_grad with two optional cudaEvent_t handles (NULL = not recorded):
 * main_start is recorded on `stream` just before the first launch of the main
 * backward kernel and main_stop just after its last one, so a caller can time
 * the dominant kernel alone with cudaEventElapsedTime.  When dQ is formed by
 * the fixed-order pass (sag_plan_info.dq_path 1 or 2), the main kernel and the
 * pass alternate per token chunk and main_stop follows the last pass.
 * Arguments, ownership and errors are those of sel_attn_grad.
 */
sag_status sel_attn_grad_timed(const sag_desc *desc, const void *query, const void *key,
                               const void *value, const void *attention_out,
                               const void *attention_out_grad, const float *softmax_max,
                               const float *softmax_sum, const int32_t *topk_indices, void *dq,
                               void *dk, void *dv, void *workspace, size_t workspace_bytes,
                               void *stream, void *main_start, void *main_stop);

/*
 * Allocation-free variant of sel_attn_grad.  The operator pages have no
 * counterpart: it exists for callers that cannot allocate device memory at
 * the point of the call -- code that runs inside a framework whose memory
 * pool forbids raw cudaMalloc, plug-ins that are handed only tensors by their
 * host, or steps where an allocation (and the synchronisation it implies) is
 * not allowed.
 *
 * The caller passes inputs, outputs and a stream as for sel_attn_grad, but no
 * workspace: the scratch lives in one fixed array of
 * SEL_ATTN_GRAD_NOALLOC_MAX_SCRATCH bytes inside the library, which every GPU
 * that loads the library holds until the process exits.  Nothing is
 * allocated, on the host or the device, by this call.
 *   - A problem whose phase-1 workspace size exceeds the maximum is rejected
 *     with SAG_ERR_WORKSPACE before anything is enqueued (use sel_attn_grad
 *     with a caller-owned workspace for those).
 *   - The first call on a device looks up that device's copy of the array
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - All calls on a device share the one array.  Each call re-initialises
 *     what has to start at zero, so earlier contents do not matter, but calls
 *     whose work overlaps on the GPU (different streams, or another thread)
 *     race on it: serialise them.
 *   - The device status (SAG_ERR_INDEX, ...) lives in the fixed array:
 *     sel_attn_grad_noalloc_query_error reads it.
 * Returns the statuses of sel_attn_grad, or SAG_ERR_WORKSPACE as above.
 */
#define SEL_ATTN_GRAD_NOALLOC_MAX_SCRATCH ((size_t)64 << 20)

sag_status sel_attn_grad_noalloc(const sag_desc *desc, const void *query, const void *key,
                                 const void *value, const void *attention_out,
                                 const void *attention_out_grad, const float *softmax_max,
                                 const float *softmax_sum, const int32_t *topk_indices, void *dq,
                                 void *dk, void *dv, void *stream);

/*
 * sel_attn_grad_query_error for the allocation-free path: synchronises
 * `stream` and returns the device-recorded status of the last
 * sel_attn_grad_noalloc on the stream's device (SAG_OK, SAG_ERR_INDEX,
 * SAG_ERR_TIMEOUT), or SAG_ERR_CUDA.  The status is that of the shared array:
 * with overlapping calls it belongs to whichever wrote it last.
 */
sag_status sel_attn_grad_noalloc_query_error(void *stream);

/*
 * Forward of selected attention: the step before the backward, producing the
 * attention_out, softmax_max and softmax_sum it takes ("NsaSelectedAttention-
 * Grad" README, parameter table: the forward's outputs; the attention is the
 * softmax(scale Q Ksel^T) Vsel of its function description over the rows the
 * Gather formula selects, and the statistics follow the FlashAttention
 * convention of "aclnnFlashAttentionUnpaddingScoreGradV3": the maximum of the
 * scaled scores and the sum of exp(score - maximum)).
 *
 * Phase 1 (host only): validates `desc` as sel_attn_grad_workspace_size does
 * and writes the forward's workspace size.  The forward runs on the tensor
 * cores only: d_v == 128, d_qk in {128, 192}, block_size in {16, 32, 48, 64,
 * 128}; other shapes return SAG_ERR_UNSUPPORTED, and so does
 * desc->deterministic == 1 (the sums and O are reduced in an order that
 * varies from run to run; the maxima are exact in any order).
 */
sag_status sel_attn_fwd_workspace_size(const sag_desc *desc, size_t *workspace_bytes);

/*
 * Phase 2: enqueues the forward on `stream` and returns without waiting.
 *   query          [T1, n1, d_qk]          dtype
 *   key            [T2, n2, d_qk]          dtype
 *   value          [T2, n2, d_v]           dtype
 *   topk_indices   [T1, n2, block_count]   int32, block ids local to the
 *                  token's batch (as for sel_attn_grad)
 *   attention_out  [T1, n1, d_v]           dtype, written
 *   softmax_max    [T1, n1, 8]             fp32, written (8 equal lanes)
 *   softmax_sum    [T1, n1, 8]             fp32, written (8 equal lanes)
 *   workspace      device scratch of at least the forward's phase-1 size
 * All pointers are device pointers, 16-byte aligned; the caller owns every
 * buffer.  Returns SAG_OK once enqueued, a host-side status (nothing
 * enqueued), or SAG_ERR_CUDA when a launch failed; out-of-range block ids are
 * recorded on the device (sel_attn_grad_query_error) and skipped.
 */
sag_status sel_attn_fwd(const sag_desc *desc, const void *query, const void *key, const void *value,
                        const int32_t *topk_indices, void *attention_out, float *softmax_max,
                        float *softmax_sum, void *workspace, size_t workspace_bytes, void *stream);

/*
 * sel_attn_fwd with two optional cudaEvent_t handles recorded just before
 * the first and just after the second tensor-core pass (NULL = not recorded).
 */
sag_status sel_attn_fwd_timed(const sag_desc *desc, const void *query, const void *key,
                              const void *value, const int32_t *topk_indices, void *attention_out,
                              float *softmax_max, float *softmax_sum, void *workspace,
                              size_t workspace_bytes, void *stream, void *passes_start,
                              void *passes_stop);

/*
 * Forward phase 2 with the tensors in one sag_io: reads query, key, value,
 * topk_indices (and query_rope, key_rope when d_rope), writes attention_out,
 * softmax_max and softmax_sum (padding rows of BSND get zeros in all three);
 * optional cudaEvent_t handles as in sel_attn_fwd_timed.  Statuses as for
 * sel_attn_fwd.
 */
sag_status sel_attn_fwd_ex(const sag_desc *desc, const sag_io *io, void *workspace, size_t workspace_bytes,
                           void *stream, void *passes_start, void *passes_stop);

/*
 * Lightning-indexer backward ("aclnnLightningIndexerGrad", formula section):
 *     S  = Relu(Matmul(Query, Gather(Key, Indices)))
 *     Y  = Dy * Weights
 *     dW = Reduce(S * dy)
 *     dQ = Matmul(ReluGrad(Y, S), Gather(Key, Indices))
 *     dK = ScatterAdd(Matmul(ReluGrad(Y, S), Q), Indices)
 * i.e. with G = n1 / n2 query heads per key head (h uses key head h / G):
 *     S[t,h,j] = relu(<q[t,h], k[idx[t,n2,j]]>)        (no scale)
 *     R[t,h,j] = dy[t,n2,j] * w[t,h] where S[t,h,j] > 0, else 0
 *     dW[t,h]  = sum_j S[t,h,j] * dy[t,n2,j]
 *     dQ[t,h]  = sum_j R[t,h,j] * k[idx[t,n2,j]]
 *     dK[idx[t,n2,j]] += sum_h R[t,h,j] * q[t,h]      (a position named twice adds twice)
 * The page's parameter tables are lost; the shapes are this library's reading.
 *
 *   batch, layout, cu_seqlens_q / cu_seqlens_kv, s1_max / s2_max: as in
 *                 sag_desc (TND, or BSND padded to s1_max / s2_max rows)
 *   n1, n2        query heads and key heads (n1 % n2 == 0, G = n1 / n2 <= 64)
 *   d             head dim of query and key (128)
 *   topk          selections per (query token, key head), >= 1; every batch's
 *                 key length is >= topk
 *   dtype         SAG_BF16 / SAG_FP16 of query, key, weights, dq, dk, dweights
 *   deterministic must be 0 (a bitwise-reproducible mode is not built: dK and
 *                 dW are summed with fp32 atomics)
 */
typedef struct sli_desc {
    int32_t batch;
    int32_t n1, n2;
    int32_t d;
    int32_t topk;
    int32_t dtype;
    int32_t deterministic;
    int32_t layout;
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_kv;
    int32_t s1_max, s2_max;
} sli_desc;

/*
 * Tensors (device pointers, 16-byte aligned, dense; R1 / R2 rows as in sag_io):
 *   query     [R1, n1, d]     dtype
 *   key       [R2, n2, d]     dtype
 *   weights   [R1, n1]        dtype
 *   dy        [R1, n2, topk]  fp32: gradient of the index score at each selection
 *   indices   [R1, n2, topk]  int32 key positions local to the token's batch;
 *                             -1 marks an empty slot (skipped); any other id
 *                             outside [0, S2_b) is reported (SAG_ERR_INDEX) and
 *                             skipped
 *   dq        [R1, n1, d], dk [R2, n2, d], dweights [R1, n1]: written (padding
 *             rows and key rows nobody selected get zeros)
 */
typedef struct sli_io {
    const void *query, *key, *weights;
    const float *dy;
    const int32_t *indices;
    void *dq, *dk, *dweights;
} sli_io;

/* Phase 1 (host only): validation and workspace size.  SAG_ERR_UNSUPPORTED for
 * d != 128, G > 64 or deterministic == 1. */
sag_status lightning_indexer_grad_workspace_size(const sli_desc *desc, size_t *workspace_bytes);

/* Phase 2: enqueue on `stream`; ownership, errors and device status as for
 * sel_attn_grad (sel_attn_grad_query_error reads this call's workspace). */
sag_status lightning_indexer_grad(const sli_desc *desc, const sli_io *io, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Self-test of the device failure path (not part of the operator; the pages
 * have no counterpart).  Enqueues one small kernel that runs the library's
 * bounded mbarrier wait on a barrier nothing ever arrives on: after limit_ns
 * (1 us .. 4 s) the wait gives up, SAG_ERR_TIMEOUT is recorded in the first
 * 256 bytes of `workspace` (device memory, 16-byte aligned, at least 256
 * bytes) and the kernel returns, so the context stays usable.  Read the
 * status back with sel_attn_grad_query_error(workspace, stream).  Returns
 * SAG_OK once enqueued, SAG_ERR_NULL / SAG_ERR_ALIGN / SAG_ERR_SHAPE for bad
 * arguments, SAG_ERR_CUDA if the launch failed.
 */
sag_status sel_attn_selftest_wait_timeout(void *workspace, uint64_t limit_ns, void *stream);

/* Static, human-readable name of a status code. */
const char *sel_attn_grad_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SELATTN_H */
