// C ABI: parameter validation (phase 1), workspace carving and the launch
// sequence (phase 2).  The parameter and shape rules follow the constraints
// section of the "NsaSelectedAttentionGrad" README; the two-phase shape
// follows the aclnn calling convention described on the same pages
// (GetWorkspaceSize validates, the second call runs on a stream).
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "kernels.cuh"

namespace sag {

namespace {

constexpr int64_t kMaxTokens = 2LL * 1024 * 1024;     // T1, T2, B <= 2M
constexpr int64_t kMaxSeq = 128LL * 1024;             // per-batch S <= 128K
constexpr size_t kAlign = 256;
// deterministic mode stores dS for at most this many bytes of query tokens at
// once; larger problems run in token chunks
constexpr int64_t kDsChunkBytes = 16LL << 30;
// total selections T1 * N2 * count the 32-bit inverted index can hold
constexpr int64_t kMaxSelections = INT32_MAX;
// default mode: token windows are sized so one (batch, KV head) window's fp32
// dQ rows take about this many bytes (they must stay resident in L2 while its
// key tiles are processed); problems whose whole dQ accumulator is smaller
// than kWindowMinAcc run without windows
constexpr int64_t kWindowDqBytes = 48LL << 20;
// Windows are built but off by default: on GB300 they measured slower than a
// single pass (the per-window key-tile reloads cost more than the L2 hits of
// the dQ reductions gained); SELATTN_WINDOW_TOKENS turns them on.
constexpr int64_t kWindowMinAcc = INT64_MAX;
// forward: no per-window dK / dV partials, so windows are on whenever the fp32
// O accumulator is well beyond L2, sized to about kFwdWindowBytes of O rows
// (measured on GB300: long-context 9.6 -> 8.6 ms, max-selection 1.05 -> 0.85 s;
// SELATTN_FWD_WINDOW_TOKENS sets the length, -1 turns them off)
constexpr int64_t kFwdWindowMinAcc = 256LL << 20;
constexpr int64_t kFwdWindowBytes = 32LL << 20;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Default mode: reduce dQ with fp32 atomics inside the main kernel, or store
// dS and form dQ by the fixed-order pass.  Bytes moved per query row:
//   reductions: count * halves * d_qk * 4 (one fp32 partial per 64-key tile)
//   dS pass:    count * bs * 2 * 2 (dS out and back) + count * bs * d_qk * 2 / G
//               (every selected key block re-read per (token, KV head))
// For the tensor-core kernel of the larger query groups (G >= 8), with
// blocks of 64 or 128 keys (the tensor-core dQ pass), the pass is
// taken when it moves less than 3x the reductions' bytes counted once per
// selected block: the 64-key tiles of a larger block reduce into the same
// rows back to back and measure like one, and the pass's key re-reads are
// served from L2.  Measured on GB300 (the main kernel storing dS with two
// query tiles in flight): 64-key blocks with G = 16 (ratio 2.33) 9.93 ms with
// the reductions, 9.15 ms with the pass; 128-key blocks with G = 32 (ratio
// 2.67) 954 ms against 919 ms.  Elsewhere (the split schedule of the small
// groups, the CUDA-core kernel, the CUDA-core dQ pass of other block sizes)
// it is taken only when it moves less than half the reductions' bytes.
// SELATTN_DQ_PASS=0 / 1 forces either.
bool prefer_dq_pass(const Geometry &g, bool main_tc_kernel) {
    const char *env = getenv("SELATTN_DQ_PASS");
    if (env && env[0] == '0') return false;
    if (env && env[0] == '1') return true;
    const double red = (double)g.block_count * g.d_qk * 4;
    const double pass = (double)g.block_count * g.block_size * 4 + (double)g.block_count * g.block_size * g.d_qk * 2 / g.group;
    return main_tc_kernel ? pass < 3.0 * red : pass < 0.5 * red * g.halves;
}

// Fixed-order dQ from per-slot partials instead of the stored dS, per query row:
//   dS pass:  count * bs * 2 * 2 + count * bs * d_qk * 2 / G (as above)
//   partials: count * halves * d_qk * 4 * 2 (each key tile's fp32 dQ partial
//             stored by the main kernel, read back once by the summing pass)
// taken when the partials move less than half the bytes: small blocks and
// small query groups, where the dS pass re-reads every selected key block per
// (token, KV head).  SELATTN_DQ_SLOTS=0 / 1 forces either.
bool prefer_dq_slots(const Geometry &g) {
    const char *env = getenv("SELATTN_DQ_SLOTS");
    if (env && env[0] == '0') return false;
    if (env && env[0] == '1') return true;
    const double slots = (double)g.block_count * g.halves * g.d_qk * 4 * 2;
    const double pass = (double)g.block_count * g.block_size * 4 + (double)g.block_count * g.block_size * g.d_qk * 2 / g.group;
    return slots < 0.5 * pass;
}

struct Plan {
    Geometry g;
    bool fp16, det;
    bool ds_path;                     // dQ by a fixed-order pass after the main kernel (else fp32 reductions)
    bool slot_path;                   // ... summing per-slot dQ partials (else from the stored dS)
    // byte offsets inside the workspace
    size_t o_hdr, o_cu_q, o_cu_kv, o_item_base, o_unit_base, o_wtab_base, o_count, o_offset, o_cursor, o_scan,
        o_entries, o_wtab, o_delta, o_lse2, o_dq_acc, o_ds, o_dkv, total;
    int32_t chunk_tokens, n_chunks;
    bool use_tc;                      // tensor-core main kernel (else the CUDA-core one)
    size_t o_q_end, o_kv_blocks;
    std::vector<int32_t> row_q;       // host copy, B+1: first query row of each batch
    std::vector<int32_t> row_kv;      // host copy, B+1: first key row of each batch
    std::vector<int32_t> q_end;       // host copy, B: end of the valid query rows
    std::vector<int32_t> kv_blocks;   // host copy, B: valid key blocks
    std::vector<int64_t> item_base;   // host copy, B+1
    std::vector<int64_t> unit_base;   // host copy, B+1 (windowed)
    std::vector<int64_t> wtab_base;   // host copy, B+1 (windowed)
};

sag_status validate(const sag_desc *d) {
    if (!d || !d->cu_seqlens_q || !d->cu_seqlens_kv) return SAG_ERR_NULL;
    if (d->dtype != SAG_BF16 && d->dtype != SAG_FP16) return SAG_ERR_DTYPE;
    if (d->reserved_ != 0 || (d->deterministic != 0 && d->deterministic != 1)) return SAG_ERR_SHAPE;
    if (d->layout != SAG_LAYOUT_TND && d->layout != SAG_LAYOUT_BSND) return SAG_ERR_SHAPE;
    if (d->batch < 1 || d->batch > kMaxTokens) return SAG_ERR_SHAPE;
    if (d->n1 < 1 || d->n1 > 128 || d->n2 < 1 || d->n2 > 128 || d->n1 % d->n2 != 0) return SAG_ERR_SHAPE;
    if (d->n1 / d->n2 > 32) return SAG_ERR_SHAPE;
    if (d->d_rope != 0 && d->d_rope != 64) return SAG_ERR_SHAPE;
    const int d_qk = d->d_qk + d->d_rope;     // head dim of the attention
    if ((d_qk != 128 && d_qk != 192) || (d->d_v != 128 && d->d_v != 192)) return SAG_ERR_SHAPE;
    // the rope split is built for the tensor-core kernels' 128 + 64 layout
    if (d->d_rope && (d->d_qk != 128 || d->d_v != 128)) return SAG_ERR_UNSUPPORTED;
    if (d->block_size < 16 || d->block_size > 128 || d->block_size % 16 != 0) return SAG_ERR_SHAPE;
    if (d->block_count < 1 || d->block_count > 128) return SAG_ERR_SHAPE;
    if ((int64_t)d->block_size * d->block_count >= 8192) return SAG_ERR_SHAPE;
    if (!(d->scale == d->scale) || d->scale > 1e30 || d->scale < -1e30) return SAG_ERR_SHAPE;
    const bool bsnd = d->layout == SAG_LAYOUT_BSND;
    if (bsnd) {
        if (d->s1_max < 1 || d->s1_max > kMaxSeq || d->s2_max < 1 || d->s2_max > kMaxSeq) return SAG_ERR_SHAPE;
        if (d->s2_max % d->block_size != 0) return SAG_ERR_SHAPE;
        if ((int64_t)d->batch * d->s1_max > kMaxTokens || (int64_t)d->batch * d->s2_max > kMaxTokens)
            return SAG_ERR_SHAPE;
    } else if (d->s1_max != 0 || d->s2_max != 0) {
        return SAG_ERR_SHAPE;
    }
    const int32_t *cq = d->cu_seqlens_q, *ck = d->cu_seqlens_kv;
    if (cq[0] != 0 || ck[0] != 0) return SAG_ERR_SHAPE;
    const int64_t sel = (int64_t)d->block_size * d->block_count;
    for (int b = 0; b < d->batch; ++b) {
        const int64_t s1 = (int64_t)cq[b + 1] - cq[b];
        const int64_t s2 = (int64_t)ck[b + 1] - ck[b];
        if (s1 < 0 || s1 > (bsnd ? d->s1_max : kMaxSeq)) return SAG_ERR_SHAPE;
        if (s2 < sel || s2 > (bsnd ? d->s2_max : kMaxSeq) || s2 % d->block_size != 0) return SAG_ERR_SHAPE;
    }
    const int64_t t1 = cq[d->batch], t2 = ck[d->batch];
    if (t1 < 1 || t1 > kMaxTokens || t2 < 1 || t2 > kMaxTokens) return SAG_ERR_SHAPE;
    return SAG_OK;
}

// forward: the same carve (dq_acc holds O, lse2 the row maxima, delta the
// row sums); tensor-core shapes only, no token windows or chunks
sag_status make_plan(const sag_desc *d, Plan *p, bool forward = false) {
    sag_status st = validate(d);
    if (st != SAG_OK) return st;
    Geometry &g = p->g;
    const bool bsnd = d->layout == SAG_LAYOUT_BSND;
    g.batch = d->batch;
    // rows of the tensors: packed (TND) or every batch padded to s*_max (BSND)
    p->row_q.assign(d->batch + 1, 0);
    p->row_kv.assign(d->batch + 1, 0);
    p->q_end.assign(d->batch, 0);
    p->kv_blocks.assign(d->batch, 0);
    for (int b = 0; b <= d->batch; ++b) {
        p->row_q[b] = bsnd ? b * d->s1_max : d->cu_seqlens_q[b];
        p->row_kv[b] = bsnd ? b * d->s2_max : d->cu_seqlens_kv[b];
    }
    for (int b = 0; b < d->batch; ++b) {
        p->q_end[b] = p->row_q[b] + (d->cu_seqlens_q[b + 1] - d->cu_seqlens_q[b]);
        p->kv_blocks[b] = (d->cu_seqlens_kv[b + 1] - d->cu_seqlens_kv[b]) / d->block_size;
    }
    g.t1 = p->row_q[d->batch];
    g.t2 = p->row_kv[d->batch];
    g.n1 = d->n1;
    g.n2 = d->n2;
    g.group = d->n1 / d->n2;
    g.d_rope = d->d_rope;
    g.d_qk = d->d_qk + d->d_rope;
    g.d_v = d->d_v;
    g.block_size = d->block_size;
    g.block_count = d->block_count;
    g.scale = (float)d->scale;
    g.scale_log2 = (float)(d->scale * 1.4426950408889634);
    p->fp16 = d->dtype == SAG_FP16;
    p->det = d->deterministic != 0;
    p->ds_path = p->det;
    p->item_base.assign(d->batch + 1, 0);
    for (int b = 0; b < d->batch; ++b) {
        // every block of the (padded) key rows is an item: blocks no token may
        // select (BSND padding) get empty buckets and zero gradients
        const int64_t nblk = (p->row_kv[b + 1] - p->row_kv[b]) / d->block_size;
        p->item_base[b + 1] = p->item_base[b] + nblk * d->n2;
    }
    g.n_items = p->item_base[d->batch];
    if (g.n_items > max_scannable_items()) return SAG_ERR_UNSUPPORTED;

    const int64_t rows = (int64_t)g.t1 * g.n1;
    const int64_t sel = (int64_t)g.t1 * g.n2 * g.block_count;
    // bucket offsets and positions inside the inverted index are 32-bit
    if (sel > kMaxSelections) return SAG_ERR_UNSUPPORTED;
    // SELATTN_FORCE_CUDA_CORE=1 selects the CUDA-core kernel for shapes the
    // tensor-core one also covers (used to cross-check the two)
    const char *force = getenv("SELATTN_FORCE_CUDA_CORE");
    p->use_tc = bwd_tc_supported(g) && !(force && force[0] == '1');
    if (g.d_rope && !p->use_tc) return SAG_ERR_UNSUPPORTED;
    if (forward) {
        if (p->det) return SAG_ERR_UNSUPPORTED;   // the forward's sums are order-dependent
        p->use_tc = fwd_tc_supported(g);
        if (!p->use_tc) return SAG_ERR_UNSUPPORTED;
    }
    g.halves = g.block_size > 64 ? g.block_size / 64 : 1;
    g.dq_slots = 0;
    // token windows: tensor-core default mode on problems whose dQ accumulator
    // is well beyond L2.  SELATTN_WINDOW_TOKENS sets the window length (and
    // forces windows on smaller problems too).
    const char *wenv = getenv(forward ? "SELATTN_FWD_WINDOW_TOKENS" : "SELATTN_WINDOW_TOKENS");
    const int acc_cols = forward ? g.d_v : g.d_qk;
    if (!forward && !p->det)
        p->ds_path = prefer_dq_pass(g, p->use_tc && !bwd_split_preferred(g) && dq_tc_supported(g));
    p->slot_path = !forward && p->ds_path && p->use_tc && prefer_dq_slots(g);
    g.dq_slots = p->slot_path ? 1 : 0;
    g.windowed = p->use_tc && !p->ds_path &&
                 (rows * acc_cols * 4 > (forward ? kFwdWindowMinAcc : kWindowMinAcc) || (wenv && atoll(wenv) > 0));
    if (wenv && atoll(wenv) < 0) g.windowed = false;
    {
        int64_t wtok = (forward ? kFwdWindowBytes : kWindowDqBytes) / ((int64_t)g.group * acc_cols * 4);
        if (wenv && atoll(wenv) > 0) wtok = atoll(wenv);
        if (wtok < 1) wtok = 1;
        if (wtok > kMaxSeq) wtok = kMaxSeq;
        g.window = (int32_t)wtok;
    }
    g.n_units = g.n_items * g.halves;
    p->unit_base.assign(d->batch + 1, 0);
    p->wtab_base.assign(d->batch + 1, 0);
    if (g.windowed) {
        for (int b = 0; b < d->batch; ++b) {
            const int64_t s1 = p->row_q[b + 1] - p->row_q[b];
            const int64_t nwin = (s1 + g.window - 1) / g.window;
            const int64_t items_b = p->item_base[b + 1] - p->item_base[b];
            p->unit_base[b + 1] = p->unit_base[b] + nwin * items_b * g.halves;
            p->wtab_base[b + 1] = p->wtab_base[b] + items_b * (nwin + 1);
        }
        g.n_units = p->unit_base[d->batch];
    }
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
    p->o_hdr = take(sizeof(WsHeader));
    p->o_cu_q = take(sizeof(int32_t) * (g.batch + 1));
    p->o_cu_kv = take(sizeof(int32_t) * (g.batch + 1));
    p->o_item_base = take(sizeof(int64_t) * (g.batch + 1));
    p->o_unit_base = take(sizeof(int64_t) * (g.batch + 1));
    p->o_wtab_base = take(sizeof(int64_t) * (g.batch + 1));
    p->o_q_end = take(sizeof(int32_t) * g.batch);
    p->o_kv_blocks = take(sizeof(int32_t) * g.batch);
    p->o_count = take(sizeof(int32_t) * (g.n_items + 1));
    p->o_cursor = take(sizeof(int32_t) * g.n_items);
    p->o_offset = take(sizeof(int32_t) * (g.n_items + 1));
    p->o_scan = take(sizeof(int32_t) * scan_parts(g.n_items));
    p->o_entries = take(sizeof(int32_t) * sel);
    p->o_wtab = take(sizeof(int32_t) * (p->wtab_base.empty() ? 0 : p->wtab_base[g.batch]));
    p->o_delta = take(sizeof(float) * rows);
    p->o_lse2 = take(sizeof(float) * rows);
    p->o_dq_acc = p->ds_path ? o : take(sizeof(float) * rows * g.d_qk);
    const int64_t ds_per_token = p->slot_path
                                     ? (int64_t)g.n1 * g.block_count * g.halves * g.d_qk * 4
                                     : (int64_t)g.n2 * g.block_count * g.group * g.block_size * 2;
    int64_t chunk = kDsChunkBytes / ds_per_token;
    // SELATTN_DS_CHUNK_TOKENS sets the chunk length (tests run the chunked
    // path on small problems with it)
    const char *cenv = getenv("SELATTN_DS_CHUNK_TOKENS");
    if (cenv && atoll(cenv) > 0) chunk = atoll(cenv);
    if (chunk < 1) chunk = 1;
    if (chunk > g.t1) chunk = g.t1;
    p->chunk_tokens = p->ds_path ? (int32_t)chunk : g.t1;
    p->n_chunks = p->ds_path ? (int32_t)((g.t1 + chunk - 1) / chunk) : 1;
    p->o_ds = p->ds_path ? take((size_t)ds_per_token * chunk) : o;
    p->o_dkv = (p->n_chunks > 1 || g.windowed) ? take(sizeof(float) * (int64_t)g.t2 * g.n2 * (g.d_qk + g.d_v)) : o;
    g.tok_lo = 0;
    g.tok_hi = g.t1;
    g.chunked = p->n_chunks > 1;
    p->total = o;
    return SAG_OK;
}

// Buckets are sorted by token where their order matters: the deterministic
// mode (dK / dV accumulated in a fixed order), token chunks and token windows
// (their ranges are found by token).  The default mode's dQ pass reads dS by
// (token, slot), whatever the order in which the main kernel wrote it.
bool buckets_sorted(const Plan &p) { return p.det || p.n_chunks > 1 || p.g.windowed; }

Workspace carve(const Plan &p, void *base) {
    char *c = static_cast<char *>(base);
    Workspace w;
    w.hdr = reinterpret_cast<WsHeader *>(c + p.o_hdr);
    w.cu_q = reinterpret_cast<int32_t *>(c + p.o_cu_q);
    w.cu_kv = reinterpret_cast<int32_t *>(c + p.o_cu_kv);
    w.q_end = reinterpret_cast<int32_t *>(c + p.o_q_end);
    w.kv_blocks = reinterpret_cast<int32_t *>(c + p.o_kv_blocks);
    w.item_base = reinterpret_cast<int64_t *>(c + p.o_item_base);
    w.count = reinterpret_cast<int32_t *>(c + p.o_count);
    w.offset = reinterpret_cast<int32_t *>(c + p.o_offset);
    w.cursor = reinterpret_cast<int32_t *>(c + p.o_cursor);
    w.scan_part = reinterpret_cast<int32_t *>(c + p.o_scan);
    w.entries = reinterpret_cast<int32_t *>(c + p.o_entries);
    w.delta = reinterpret_cast<float *>(c + p.o_delta);
    w.lse2 = reinterpret_cast<float *>(c + p.o_lse2);
    w.dq_acc = p.ds_path ? nullptr : reinterpret_cast<float *>(c + p.o_dq_acc);
    w.ds = (p.ds_path && !p.slot_path) ? reinterpret_cast<uint16_t *>(c + p.o_ds) : nullptr;
    w.dq_part = p.slot_path ? reinterpret_cast<float *>(c + p.o_ds) : nullptr;
    w.dkv_acc = (p.n_chunks > 1 || p.g.windowed) ? reinterpret_cast<float *>(c + p.o_dkv) : nullptr;
    w.unit_base = reinterpret_cast<int64_t *>(c + p.o_unit_base);
    w.wtab_base = reinterpret_cast<int64_t *>(c + p.o_wtab_base);
    w.wtab = reinterpret_cast<int32_t *>(c + p.o_wtab);
    return w;
}

bool aligned16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; }

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return sms;
}

}  // namespace

bool DeviceGuard::bind(cudaStream_t s) {
    if (s == nullptr) return true;
    int dev = 0;
    if (cudaStreamGetDevice(s, &dev) != cudaSuccess) return false;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    if (cur == dev) return true;
    if (cudaSetDevice(dev) != cudaSuccess) return false;
    saved_ = cur;
    return true;
}

DeviceGuard::~DeviceGuard() {
    if (saved_ >= 0) cudaSetDevice(saved_);
}

}  // namespace sag

using namespace sag;

extern "C" sag_status sel_attn_grad_workspace_size(const sag_desc *desc, size_t *workspace_bytes) {
    if (!workspace_bytes) return SAG_ERR_NULL;
    Plan p;
    sag_status st = make_plan(desc, &p);
    if (st != SAG_OK) return st;
    *workspace_bytes = p.total;
    return SAG_OK;
}

namespace {
int launches_of(const Plan &p) {
    // preprocess, histogram, 3 scan passes, fill (, sort)
    int n = 6 + (buckets_sorted(p) ? 1 : 0);
    if (!p.ds_path) return n + 2 + (p.g.windowed ? 1 : 0);   // main, cast dQ (, cast dK/dV)
    return n + 2 * p.n_chunks + (p.n_chunks > 1);    // (main, dQ) per chunk, cast dK/dV
}
}  // namespace

extern "C" sag_status sel_attn_grad_plan_info(const sag_desc *desc, sag_plan_info *info) {
    if (!info) return SAG_ERR_NULL;
    Plan p;
    sag_status st = make_plan(desc, &p);
    if (st != SAG_OK) return st;
    info->workspace_bytes = p.total;
    info->launches = launches_of(p);
    info->token_chunks = p.n_chunks;
    info->items = p.g.n_items;
    info->main_kernel = p.use_tc ? 1 : 0;
    info->dq_path = p.slot_path ? 2 : p.ds_path ? 1 : 0;
    return SAG_OK;
}

namespace {

// Checks shared by the backward and the forward: required pointers,
// alignment, workspace size.
sag_status check_io(const Plan &p, const void *const *ptrs, int n, const sag_io *io, void *workspace,
                    size_t workspace_bytes) {
    for (int i = 0; i < n; ++i)
        if (!ptrs[i]) return SAG_ERR_NULL;
    if (p.g.d_rope && (!io->query_rope || !io->key_rope)) return SAG_ERR_NULL;
    if (!workspace) return SAG_ERR_WORKSPACE;
    for (int i = 0; i < n; ++i)
        if (!aligned16(ptrs[i])) return SAG_ERR_ALIGN;
    if (p.g.d_rope && (!aligned16(io->query_rope) || !aligned16(io->key_rope))) return SAG_ERR_ALIGN;
    if (!aligned16(workspace)) return SAG_ERR_ALIGN;
    if (workspace_bytes < p.total) return SAG_ERR_WORKSPACE;
    return SAG_OK;
}

// Header reset, the host metadata copy (row starts, valid ends, item and
// window bases) and the bucket counters' memset.  The host buffer is
// pageable: the copy has consumed it by the time cudaMemcpyAsync returns.
sag_status stage_metadata(const Plan &p, void *workspace, cudaStream_t s) {
    const Geometry &g = p.g;
    std::vector<char> meta(p.o_count - p.o_cu_q, 0);
    auto put = [&](size_t off, const void *src, size_t bytes) { memcpy(meta.data() + (off - p.o_cu_q), src, bytes); };
    put(p.o_cu_q, p.row_q.data(), sizeof(int32_t) * (g.batch + 1));
    put(p.o_cu_kv, p.row_kv.data(), sizeof(int32_t) * (g.batch + 1));
    put(p.o_item_base, p.item_base.data(), sizeof(int64_t) * (g.batch + 1));
    put(p.o_unit_base, p.unit_base.data(), sizeof(int64_t) * (g.batch + 1));
    put(p.o_wtab_base, p.wtab_base.data(), sizeof(int64_t) * (g.batch + 1));
    put(p.o_q_end, p.q_end.data(), sizeof(int32_t) * g.batch);
    put(p.o_kv_blocks, p.kv_blocks.data(), sizeof(int32_t) * g.batch);
    char *base = static_cast<char *>(workspace);
    if (cudaMemsetAsync(base + p.o_hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return SAG_ERR_CUDA;
    if (cudaMemcpyAsync(base + p.o_cu_q, meta.data(), meta.size(), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return SAG_ERR_CUDA;
    // count and cursor are adjacent: one memset
    if (cudaMemsetAsync(base + p.o_count, 0, p.o_offset - p.o_count, s) != cudaSuccess) return SAG_ERR_CUDA;
    return SAG_OK;
}

cudaError_t launch_main(const Plan &p, const Geometry &g, const Workspace &ws, const sag_io &io, bool det,
                        cudaStream_t s, int sms) {
    if (!p.use_tc) return launch_bwd_simt(g, ws, io, p.fp16, det, s, sms);
    if (bwd_split_preferred(g)) return launch_bwd_tc_split(g, ws, io, p.fp16, det, s, sms);
    return launch_bwd_tc(g, ws, io, p.fp16, det, s, sms);
}

}  // namespace

extern "C" sag_status sel_attn_grad(const sag_desc *desc, const void *query, const void *key,
                                    const void *value, const void *attention_out,
                                    const void *attention_out_grad, const float *softmax_max,
                                    const float *softmax_sum, const int32_t *topk_indices, void *dq,
                                    void *dk, void *dv, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    return sel_attn_grad_timed(desc, query, key, value, attention_out, attention_out_grad, softmax_max,
                               softmax_sum, topk_indices, dq, dk, dv, workspace, workspace_bytes, stream,
                               nullptr, nullptr);
}

extern "C" sag_status sel_attn_grad_timed(const sag_desc *desc, const void *query, const void *key,
                                          const void *value, const void *attention_out,
                                          const void *attention_out_grad, const float *softmax_max,
                                          const float *softmax_sum, const int32_t *topk_indices, void *dq,
                                          void *dk, void *dv, void *workspace, size_t workspace_bytes,
                                          void *stream, void *main_start, void *main_stop) {
    sag_io io{};
    io.query = query;
    io.key = key;
    io.value = value;
    // the backward only reads these three
    io.attention_out = const_cast<void *>(attention_out);
    io.attention_out_grad = attention_out_grad;
    io.softmax_max = const_cast<float *>(softmax_max);
    io.softmax_sum = const_cast<float *>(softmax_sum);
    io.topk_indices = topk_indices;
    io.dq = dq;
    io.dk = dk;
    io.dv = dv;
    return sel_attn_grad_ex(desc, &io, workspace, workspace_bytes, stream, main_start, main_stop);
}

extern "C" sag_status sel_attn_grad_ex(const sag_desc *desc, const sag_io *io, void *workspace,
                                       size_t workspace_bytes, void *stream, void *main_start, void *main_stop) {
    cudaEvent_t ev0 = static_cast<cudaEvent_t>(main_start), ev1 = static_cast<cudaEvent_t>(main_stop);
    Plan p;
    sag_status st = make_plan(desc, &p);
    if (st != SAG_OK) return st;
    if (!io) return SAG_ERR_NULL;
    const void *ptrs[] = {io->query, io->key, io->value, io->attention_out, io->attention_out_grad, io->softmax_max,
                          io->softmax_sum, io->topk_indices, io->dq, io->dk, io->dv};
    st = check_io(p, ptrs, 11, io, workspace, workspace_bytes);
    if (st != SAG_OK) return st;
    if (p.g.d_rope && (!io->dq_rope || !io->dk_rope)) return SAG_ERR_NULL;
    if (p.g.d_rope && (!aligned16(io->dq_rope) || !aligned16(io->dk_rope))) return SAG_ERR_ALIGN;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceGuard dg;
    if (!dg.bind(s)) return SAG_ERR_CUDA;
    const Geometry &g = p.g;
    Workspace ws = carve(p, workspace);
    const int sms = device_sms();
    st = stage_metadata(p, workspace, s);
    if (st != SAG_OK) return st;

    if ((launch_preprocess(g, ws, io->attention_out, io->attention_out_grad, io->softmax_max, io->softmax_sum,
                           p.fp16, !p.ds_path, s, sms)) != cudaSuccess)
        return SAG_ERR_CUDA;
    if ((launch_inversion(g, ws, io->topk_indices, buckets_sorted(p), s, sms)) != cudaSuccess) return SAG_ERR_CUDA;
    if (!p.ds_path) {
        if (g.windowed &&
            cudaMemsetAsync(ws.dkv_acc, 0, sizeof(float) * (size_t)g.t2 * g.n2 * (g.d_qk + g.d_v), s) != cudaSuccess)
            return SAG_ERR_CUDA;
        if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return SAG_ERR_CUDA;
        if (launch_main(p, g, ws, *io, false, s, sms) != cudaSuccess) return SAG_ERR_CUDA;
        if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return SAG_ERR_CUDA;
        if ((launch_cast_dq(g, ws.dq_acc, io->dq, io->dq_rope, p.fp16, s, sms)) != cudaSuccess) return SAG_ERR_CUDA;
        if (g.windowed && (launch_cast_dkv(g, ws, io->dk, io->dk_rope, io->dv, p.fp16, s, sms)) != cudaSuccess)
            return SAG_ERR_CUDA;
        return SAG_OK;
    }
    // deterministic mode (or the dQ pass chosen for the default mode): token
    // chunks in order; dS (or the per-slot dQ partials) of a chunk -> its dQ
    if (g.chunked && cudaMemsetAsync(ws.dkv_acc, 0, sizeof(float) * (size_t)g.t2 * g.n2 * (g.d_qk + g.d_v), s) !=
                         cudaSuccess)
        return SAG_ERR_CUDA;
    if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return SAG_ERR_CUDA;
    for (int c = 0; c < p.n_chunks; ++c) {
        Geometry gc = g;
        gc.tok_lo = c * p.chunk_tokens;
        gc.tok_hi = gc.tok_lo + p.chunk_tokens < g.t1 ? gc.tok_lo + p.chunk_tokens : g.t1;
        if (launch_main(p, gc, ws, *io, true, s, sms) != cudaSuccess) return SAG_ERR_CUDA;
        const cudaError_t e = p.slot_path ? launch_dq_slots(gc, ws, *io, p.fp16, s, sms)
                              : (p.use_tc && dq_tc_supported(gc)) ? launch_dq_tc(gc, ws, *io, p.fp16, s, sms)
                                                                  : launch_dq_from_ds(gc, ws, *io, p.fp16, s, sms);
        if (e != cudaSuccess) return SAG_ERR_CUDA;
    }
    if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return SAG_ERR_CUDA;
    if (g.chunked && (launch_cast_dkv(g, ws, io->dk, io->dk_rope, io->dv, p.fp16, s, sms)) != cudaSuccess)
        return SAG_ERR_CUDA;
    return SAG_OK;
}

extern "C" sag_status sel_attn_fwd_workspace_size(const sag_desc *desc, size_t *workspace_bytes) {
    if (!workspace_bytes) return SAG_ERR_NULL;
    Plan p;
    sag_status st = make_plan(desc, &p, true);
    if (st != SAG_OK) return st;
    *workspace_bytes = p.total;
    return SAG_OK;
}

extern "C" sag_status sel_attn_fwd(const sag_desc *desc, const void *query, const void *key, const void *value,
                                   const int32_t *topk_indices, void *attention_out, float *softmax_max,
                                   float *softmax_sum, void *workspace, size_t workspace_bytes, void *stream) {
    return sel_attn_fwd_timed(desc, query, key, value, topk_indices, attention_out, softmax_max, softmax_sum,
                              workspace, workspace_bytes, stream, nullptr, nullptr);
}

extern "C" sag_status sel_attn_fwd_timed(const sag_desc *desc, const void *query, const void *key,
                                         const void *value, const int32_t *topk_indices, void *attention_out,
                                         float *softmax_max, float *softmax_sum, void *workspace,
                                         size_t workspace_bytes, void *stream, void *passes_start,
                                         void *passes_stop) {
    sag_io io{};
    io.query = query;
    io.key = key;
    io.value = value;
    io.topk_indices = topk_indices;
    io.attention_out = attention_out;
    io.softmax_max = softmax_max;
    io.softmax_sum = softmax_sum;
    return sel_attn_fwd_ex(desc, &io, workspace, workspace_bytes, stream, passes_start, passes_stop);
}

extern "C" sag_status sel_attn_fwd_ex(const sag_desc *desc, const sag_io *io, void *workspace,
                                      size_t workspace_bytes, void *stream, void *passes_start, void *passes_stop) {
    cudaEvent_t ev0 = static_cast<cudaEvent_t>(passes_start), ev1 = static_cast<cudaEvent_t>(passes_stop);
    Plan p;
    sag_status st = make_plan(desc, &p, true);
    if (st != SAG_OK) return st;
    if (!io) return SAG_ERR_NULL;
    const void *ptrs[] = {io->query, io->key, io->value, io->topk_indices, io->attention_out, io->softmax_max,
                          io->softmax_sum};
    st = check_io(p, ptrs, 7, io, workspace, workspace_bytes);
    if (st != SAG_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceGuard dg;
    if (!dg.bind(s)) return SAG_ERR_CUDA;
    const Geometry &g = p.g;
    Workspace ws = carve(p, workspace);
    const int sms = device_sms();
    st = stage_metadata(p, workspace, s);
    if (st != SAG_OK) return st;
    if (launch_fwd_init(g, ws, s, sms) != cudaSuccess) return SAG_ERR_CUDA;
    if (launch_inversion(g, ws, io->topk_indices, g.windowed, s, sms) != cudaSuccess) return SAG_ERR_CUDA;
    if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return SAG_ERR_CUDA;
    for (int pass = 1; pass <= 2; ++pass)
        if (launch_fwd_tc(g, ws, *io, pass, p.fp16, s, sms) != cudaSuccess) return SAG_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return SAG_ERR_CUDA;
    if (launch_fwd_finalize(g, ws, io->attention_out, io->softmax_max, io->softmax_sum, p.fp16, s, sms) !=
        cudaSuccess)
        return SAG_ERR_CUDA;
    return SAG_OK;
}

// ---------------------------------------------------------------------------
// Lightning-indexer backward: validation, workspace carve, launch sequence.
namespace {

struct LiPlan {
    Geometry g;
    bool fp16, bsnd;
    std::vector<int32_t> row_q, row_kv, q_end, kv_len;
    size_t o_hdr, o_cu_q, o_cu_kv, o_q_end, o_kv_len, o_dk, o_dw, total;
};

sag_status li_plan(const sli_desc *d, LiPlan *p) {
    if (!d || !d->cu_seqlens_q || !d->cu_seqlens_kv) return SAG_ERR_NULL;
    if (d->dtype != SAG_BF16 && d->dtype != SAG_FP16) return SAG_ERR_DTYPE;
    if (d->deterministic != 0 && d->deterministic != 1) return SAG_ERR_SHAPE;
    if (d->layout != SAG_LAYOUT_TND && d->layout != SAG_LAYOUT_BSND) return SAG_ERR_SHAPE;
    if (d->batch < 1 || d->batch > kMaxTokens) return SAG_ERR_SHAPE;
    if (d->n1 < 1 || d->n2 < 1 || d->n1 % d->n2 != 0 || d->d < 1 || d->topk < 1 || d->topk > kMaxSeq)
        return SAG_ERR_SHAPE;
    const bool bsnd = d->layout == SAG_LAYOUT_BSND;
    if (bsnd) {
        if (d->s1_max < 1 || d->s1_max > kMaxSeq || d->s2_max < 1 || d->s2_max > kMaxSeq) return SAG_ERR_SHAPE;
        if ((int64_t)d->batch * d->s1_max > kMaxTokens || (int64_t)d->batch * d->s2_max > kMaxTokens)
            return SAG_ERR_SHAPE;
    } else if (d->s1_max != 0 || d->s2_max != 0) {
        return SAG_ERR_SHAPE;
    }
    const int32_t *cq = d->cu_seqlens_q, *ck = d->cu_seqlens_kv;
    if (cq[0] != 0 || ck[0] != 0) return SAG_ERR_SHAPE;
    for (int b = 0; b < d->batch; ++b) {
        const int64_t s1 = (int64_t)cq[b + 1] - cq[b], s2 = (int64_t)ck[b + 1] - ck[b];
        if (s1 < 0 || s1 > (bsnd ? d->s1_max : kMaxSeq)) return SAG_ERR_SHAPE;
        if (s2 < d->topk || s2 > (bsnd ? d->s2_max : kMaxSeq)) return SAG_ERR_SHAPE;
    }
    if ((int64_t)cq[d->batch] > kMaxTokens || (int64_t)ck[d->batch] > kMaxTokens || ck[d->batch] < 1)
        return SAG_ERR_SHAPE;
    if (d->deterministic) return SAG_ERR_UNSUPPORTED;
    Geometry &g = p->g;
    g = Geometry{};
    g.batch = d->batch;
    g.n1 = d->n1;
    g.n2 = d->n2;
    g.group = d->n1 / d->n2;
    g.d_qk = d->d;
    g.block_count = d->topk;
    if (!lig_tc_supported(g)) return SAG_ERR_UNSUPPORTED;
    p->fp16 = d->dtype == SAG_FP16;
    p->bsnd = bsnd;
    p->row_q.assign(d->batch + 1, 0);
    p->row_kv.assign(d->batch + 1, 0);
    p->q_end.assign(d->batch, 0);
    p->kv_len.assign(d->batch, 0);
    for (int b = 0; b <= d->batch; ++b) {
        p->row_q[b] = bsnd ? b * d->s1_max : cq[b];
        p->row_kv[b] = bsnd ? b * d->s2_max : ck[b];
    }
    for (int b = 0; b < d->batch; ++b) {
        p->q_end[b] = p->row_q[b] + (cq[b + 1] - cq[b]);
        p->kv_len[b] = ck[b + 1] - ck[b];
    }
    g.t1 = p->row_q[d->batch];
    g.t2 = p->row_kv[d->batch];
    g.tok_hi = g.t1;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
    p->o_hdr = take(sizeof(WsHeader));
    p->o_cu_q = take(sizeof(int32_t) * (g.batch + 1));
    p->o_cu_kv = take(sizeof(int32_t) * (g.batch + 1));
    p->o_q_end = take(sizeof(int32_t) * g.batch);
    p->o_kv_len = take(sizeof(int32_t) * g.batch);
    p->o_dk = take(sizeof(float) * (size_t)g.t2 * g.n2 * g.d_qk);
    p->o_dw = take(sizeof(float) * (size_t)g.t1 * g.n1);
    p->total = o;
    return SAG_OK;
}

}  // namespace

extern "C" sag_status lightning_indexer_grad_workspace_size(const sli_desc *desc, size_t *workspace_bytes) {
    if (!workspace_bytes) return SAG_ERR_NULL;
    LiPlan p;
    sag_status st = li_plan(desc, &p);
    if (st != SAG_OK) return st;
    *workspace_bytes = p.total;
    return SAG_OK;
}

extern "C" sag_status lightning_indexer_grad(const sli_desc *desc, const sli_io *io, void *workspace,
                                             size_t workspace_bytes, void *stream) {
    LiPlan p;
    sag_status st = li_plan(desc, &p);
    if (st != SAG_OK) return st;
    if (!io) return SAG_ERR_NULL;
    const void *ptrs[] = {io->query, io->key, io->weights, io->dy, io->indices, io->dq, io->dk, io->dweights};
    for (const void *x : ptrs)
        if (!x) return SAG_ERR_NULL;
    if (!workspace) return SAG_ERR_WORKSPACE;
    for (const void *x : ptrs)
        if (!aligned16(x)) return SAG_ERR_ALIGN;
    if (!aligned16(workspace)) return SAG_ERR_ALIGN;
    if (workspace_bytes < p.total) return SAG_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceGuard dg;
    if (!dg.bind(s)) return SAG_ERR_CUDA;
    const Geometry &g = p.g;
    char *base = static_cast<char *>(workspace);
    Workspace ws{};
    ws.hdr = reinterpret_cast<WsHeader *>(base + p.o_hdr);
    ws.cu_q = reinterpret_cast<int32_t *>(base + p.o_cu_q);
    ws.cu_kv = reinterpret_cast<int32_t *>(base + p.o_cu_kv);
    ws.q_end = reinterpret_cast<int32_t *>(base + p.o_q_end);
    ws.kv_blocks = reinterpret_cast<int32_t *>(base + p.o_kv_len);
    ws.dq_acc = reinterpret_cast<float *>(base + p.o_dk);
    ws.dkv_acc = reinterpret_cast<float *>(base + p.o_dw);
    std::vector<char> meta(p.o_dk - p.o_cu_q, 0);
    auto put = [&](size_t off, const void *src, size_t bytes) { memcpy(meta.data() + (off - p.o_cu_q), src, bytes); };
    put(p.o_cu_q, p.row_q.data(), sizeof(int32_t) * (g.batch + 1));
    put(p.o_cu_kv, p.row_kv.data(), sizeof(int32_t) * (g.batch + 1));
    put(p.o_q_end, p.q_end.data(), sizeof(int32_t) * g.batch);
    put(p.o_kv_len, p.kv_len.data(), sizeof(int32_t) * g.batch);
    if (cudaMemsetAsync(base + p.o_hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return SAG_ERR_CUDA;
    if (cudaMemcpyAsync(base + p.o_cu_q, meta.data(), meta.size(), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return SAG_ERR_CUDA;
    // both fp32 accumulators are adjacent: one memset
    if (cudaMemsetAsync(base + p.o_dk, 0, p.total - p.o_dk, s) != cudaSuccess) return SAG_ERR_CUDA;
    // padding rows (BSND) of dq get no unit: zero them with the rest
    const int es = 2;
    if (p.bsnd && cudaMemsetAsync(io->dq, 0, (size_t)g.t1 * g.n1 * g.d_qk * es, s) != cudaSuccess)
        return SAG_ERR_CUDA;
    if (launch_lig(g, ws, *io, p.fp16, s, device_sms()) != cudaSuccess) return SAG_ERR_CUDA;
    return SAG_OK;
}

extern "C" sag_status sel_attn_grad_query_error(const void *workspace, void *stream) {
    if (!workspace) return SAG_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceGuard dg;
    if (!dg.bind(s)) return SAG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SAG_ERR_CUDA;
    int32_t code = 0;
    if (cudaMemcpy(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess) return SAG_ERR_CUDA;
    return static_cast<sag_status>(code);
}

extern "C" const char *sel_attn_grad_status_string(int status) {
    switch (status) {
    case SAG_OK: return "ok";
    case SAG_ERR_NULL: return "a required pointer is NULL";
    case SAG_ERR_SHAPE: return "a size or length is outside the operator's constraints";
    case SAG_ERR_DTYPE: return "dtype must be bf16 or fp16";
    case SAG_ERR_UNSUPPORTED: return "allowed by the constraints but not supported by this library";
    case SAG_ERR_WORKSPACE: return "workspace missing or smaller than the phase-1 size";
    case SAG_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
    case SAG_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case SAG_ERR_INDEX: return "a topkIndices entry is outside its batch's block range";
    case SAG_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    default: return "unknown status";
    }
}
