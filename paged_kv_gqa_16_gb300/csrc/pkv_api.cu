// pkv_api.cu -- the C ABI of libpkv (declared in include/pkv.h): argument
// checks, the split planner, the workspace layout and kernel dispatch.
// Nothing here allocates, synchronises or prints.
#include <cmath>
#include <cstdint>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {

pkv_status check_dims(const pkv_dims *d)
{
    if (d == nullptr)
        return PKV_ERR_INVALID_ARG;
    if (d->B < 0 || d->B > 65535 || d->Hq <= 0 || d->Hkv <= 0 || d->Hkv > 65535 ||
        d->page_size <= 0 || d->num_pages <= 0 || d->num_indices < 0 || d->max_seq_len < 0 ||
        d->max_seq_len > (1 << 30) || !std::isfinite(d->scale))
        return PKV_ERR_INVALID_ARG;
    if (d->Hq % d->Hkv != 0)
        return PKV_ERR_INVALID_ARG;
    if (d->D != 64 && d->D != 128)
        return PKV_ERR_UNSUPPORTED;
    if (d->Hq / d->Hkv > 16)
        return PKV_ERR_UNSUPPORTED;
    // element offsets inside a pool must fit the 64-bit arithmetic used
    if ((double)d->num_pages * d->page_size * d->Hkv * d->D > 9.0e18)
        return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

} // namespace pkv

namespace {

using pkv::check_dims;
using pkv::kMaxSplits;

constexpr size_t kHeaderBytes = 256;
constexpr int kMinChunkTokens = 256;   // per-split path: never split finer than this

size_t round_up(size_t x, size_t a)
{
    return (x + a - 1) / a * a;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

pkv_status launch_status(cudaError_t e)
{
    return e == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int chunk_for(const pkv_dims *d, int num_splits)
{
    const long long per = ((long long)d->max_seq_len + num_splits - 1) / num_splits;
    long long c = (per + 15) / 16 * 16;
    if (c < 16)
        c = 16;
    return (int)c;
}

int log2_exact(int x)
{
    if (x <= 0 || (x & (x - 1)) != 0)
        return -1;
    int s = 0;
    while ((1 << s) != x)
        ++s;
    return s;
}

// Workspace: [header 256 B | row info, persistent path: Bv x 2 int32 |
//             the per-step plan, persistent path | rotated-q scratch
//             [B, Hq, D] bf16 | one-page-per-row table of
//             the contiguous-cache call, (2B + 1) int32 | partials].
// The partial region holds either layout: the per-split one [B,Hq,S,(2|D)]
// of paged_decode_partials, or the piece one [(S+Bv)*HQV, (2|D)] of the
// persistent path.  Every region starts on a 256-byte boundary.
struct Layout {
    int hpc, Bv, HQV;
    size_t rowinfo_off, plan_off, qscratch_off, table_off, split_ml_off, split_o_off,
        piece_ml_off, piece_o_off, total;
};

Layout layout_for(const pkv_dims *d, int num_splits)
{
    Layout L{};
    L.hpc = pkv::fused_heads_per_block(d->Hkv);
    L.Bv = d->B * (d->Hkv / L.hpc);
    L.HQV = L.hpc * (d->Hq / d->Hkv);
    L.rowinfo_off = kHeaderBytes;
    L.plan_off = L.rowinfo_off + round_up((size_t)L.Bv * 2 * sizeof(int32_t), 256);
    // the per-step plan, for shapes the persistent path serves
    const size_t plan = L.Bv <= pkv::kFusedMaxRows
                            ? pkv::plan_words(L.Bv, num_splits) * sizeof(int32_t) : 0;
    L.qscratch_off = L.plan_off + round_up(plan, 256);
    L.table_off = L.qscratch_off + round_up((size_t)d->B * d->Hq * d->D * 2, 256);
    const size_t part = L.table_off + round_up(((size_t)2 * d->B + 1) * sizeof(int32_t), 256);
    const size_t rows = (size_t)d->B * d->Hq * num_splits;
    L.split_ml_off = part;
    L.split_o_off = part + round_up(rows * 2 * sizeof(float), 256);
    const size_t split_end = L.split_o_off + round_up(rows * d->D * sizeof(float), 256);
    const size_t pieces = ((size_t)num_splits + L.Bv) * L.HQV;
    L.piece_ml_off = part;
    L.piece_o_off = part + round_up(pieces * 2 * sizeof(float), 256);
    const size_t piece_end = L.piece_o_off + round_up(pieces * d->D * sizeof(float), 256);
    L.total = split_end > piece_end ? split_end : piece_end;
    return L;
}

// The persistent path keeps every virtual row's prefix sum in shared memory.
bool fused_path_ok(const pkv_dims *d)
{
    const Layout L = layout_for(d, 1);
    return L.Bv <= pkv::kFusedMaxRows &&
           (long long)L.Bv * ((long long)d->max_seq_len + pkv::kFusedRowCost) < (1ll << 31);
}

pkv_status check_decode_args(const pkv_dims *dims, const void *q, const void *k_pool,
                             const void *v_pool, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *seq_lens, int num_splits,
                             void *workspace, size_t ws_bytes, void *out, bool need_out)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (num_splits < 1 || num_splits > kMaxSplits)
        return PKV_ERR_INVALID_ARG;
    if (dims->B == 0)
        return PKV_OK;
    if (q == nullptr || k_pool == nullptr || v_pool == nullptr || kv_indptr == nullptr ||
        seq_lens == nullptr || workspace == nullptr || (need_out && out == nullptr))
        return PKV_ERR_INVALID_ARG;
    if (dims->num_indices > 0 && kv_indices == nullptr)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(workspace, 256) || (need_out && !aligned(out, 16)) ||
        !aligned(kv_indptr, 4) || !aligned(seq_lens, 4) ||
        (kv_indices != nullptr && !aligned(kv_indices, 4)))
        return PKV_ERR_INVALID_ARG;
    const size_t need = pkv_workspace_bytes(dims, num_splits);
    if (need == 0)
        return PKV_ERR_INVALID_ARG;
    if (ws_bytes < need)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    return PKV_OK;
}

// Per-(split, kv head, row) blocks: writes split partials, or the output
// directly when `direct` (one split).  Arguments already checked.
pkv_status launch_split(const pkv_dims *dims, const void *q, const void *k_pool,
                        const void *v_pool, const int32_t *kv_indices, const int32_t *kv_indptr,
                        const int32_t *seq_lens, int num_splits, void *workspace, void *out,
                        bool direct, pkv_stream_t stream)
{
    const Layout L = layout_for(dims, num_splits);
    char *ws = static_cast<char *>(workspace);
    pkv::DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_pool = static_cast<const __nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16 *>(v_pool);
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.seq_lens = seq_lens;
    p.ml_part = reinterpret_cast<float *>(ws + L.split_ml_off);
    p.o_part = reinterpret_cast<float *>(ws + L.split_o_off);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.status = reinterpret_cast<uint32_t *>(ws);
    p.B = dims->B;
    p.Hq = dims->Hq;
    p.Hkv = dims->Hkv;
    p.n_rep = dims->Hq / dims->Hkv;
    p.page_size = dims->page_size;
    p.ps_shift = log2_exact(dims->page_size);
    p.num_pages = dims->num_pages;
    p.num_indices = dims->num_indices;
    p.max_seq_len = dims->max_seq_len;
    p.num_splits = num_splits;
    p.chunk = chunk_for(dims, num_splits);
    p.direct = direct ? 1 : 0;
    p.scale_log2 = (float)((double)dims->scale * 1.4426950408889634);
    return launch_status(pkv::launch_split_decode(p, dims->D, (cudaStream_t)stream));
}

pkv_status launch_combine_split(const pkv_dims *dims, int num_splits, void *workspace,
                                void *out, pkv_stream_t stream)
{
    const Layout L = layout_for(dims, num_splits);
    char *ws = static_cast<char *>(workspace);
    pkv::CombineParams p{};
    p.o_part = reinterpret_cast<const float *>(ws + L.split_o_off);
    p.ml_part = reinterpret_cast<const float *>(ws + L.split_ml_off);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.B = dims->B;
    p.Hq = dims->Hq;
    p.D = dims->D;
    p.num_splits = num_splits;
    return launch_status(pkv::launch_combine(p, (cudaStream_t)stream));
}

// Persistent path: the token-balanced kernel, then the piece combine.  With
// k_new != nullptr the kernel also appends the step's new token (fused step).
// The persistent path's parameters (shape, tables, workspace regions).
pkv::FusedParams persistent_params(const pkv_dims *dims, const Layout &L, char *ws,
                                   const int32_t *kv_indices, const int32_t *kv_indptr,
                                   const int32_t *seq_lens)
{
    pkv::FusedParams p{};
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.seq_lens = seq_lens;
    p.row_info = reinterpret_cast<int32_t *>(ws + L.rowinfo_off);
    p.status = reinterpret_cast<uint32_t *>(ws);
    p.B = dims->B;
    p.Hq = dims->Hq;
    p.Hkv = dims->Hkv;
    p.n_rep = dims->Hq / dims->Hkv;
    p.page_size = dims->page_size;
    p.ps_shift = log2_exact(dims->page_size);
    p.num_pages = dims->num_pages;
    p.num_indices = dims->num_indices;
    p.max_seq_len = dims->max_seq_len;
    p.Bv = L.Bv;
    p.row_cost = pkv::kFusedRowCost;
    p.hpc = L.hpc;
    return p;
}

pkv_status launch_persistent(const pkv_dims *dims, const void *q, const void *k_pool,
                             const void *v_pool, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *seq_lens,
                             int num_splits, void *workspace, void *out, const void *k_new,
                             const void *v_new, const float *rope, int rope_max_pos,
                             pkv_stream_t stream, const pkv::AdvanceParams *adv = nullptr,
                             bool planned = false)
{
    const Layout L = layout_for(dims, num_splits);
    char *ws = static_cast<char *>(workspace);
    pkv::FusedParams p = persistent_params(dims, L, ws, kv_indices, kv_indptr, seq_lens);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_pool = static_cast<const __nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16 *>(v_pool);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.o_part = reinterpret_cast<float *>(ws + L.piece_o_off);
    p.ml_part = reinterpret_cast<float *>(ws + L.piece_ml_off);
    int32_t *plan_region = reinterpret_cast<int32_t *>(ws + L.plan_off);
    p.plan = planned ? plan_region : nullptr;
    p.plan_out = planned ? nullptr : plan_region;
    p.scale_log2 = (float)((double)dims->scale * 1.4426950408889634);
    p.step = k_new != nullptr ? 1 : 0;
    p.k_pool_w = const_cast<__nv_bfloat16 *>(p.k_pool);
    p.v_pool_w = const_cast<__nv_bfloat16 *>(p.v_pool);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.rope = rope;
    p.rope_max_pos = rope_max_pos;
    pkv_status st =
        launch_status(pkv::launch_fused_decode(p, dims->D, num_splits, (cudaStream_t)stream));
    if (st != PKV_OK || num_splits == 1)
        return st;
    pkv::PieceCombineParams c{};
    c.o_part = p.o_part;
    c.ml_part = p.ml_part;
    c.row_info = p.row_info;
    c.out = p.out;
    c.B = dims->B;
    c.Bv = L.Bv;
    c.Hq = dims->Hq;
    c.HQV = L.HQV;
    c.planned = planned ? 1 : 0;
    if (adv != nullptr)
        c.adv = *adv;
    return launch_status(
        pkv::launch_piece_combine(c, dims->D, num_splits, (cudaStream_t)stream));
}

pkv_status check_append_args(const pkv_dims *dims, const void *q, const void *k_new,
                             const void *v_new, const void *k_pool, const void *v_pool,
                             const int32_t *kv_indices, const int32_t *kv_indptr,
                             const int32_t *seq_lens, const float *rope_cos_sin,
                             int rope_max_pos, int rope_q, const uint32_t *status)
{
    if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr ||
        kv_indptr == nullptr || seq_lens == nullptr ||
        (dims->num_indices > 0 && kv_indices == nullptr))
        return PKV_ERR_INVALID_ARG;
    if (rope_cos_sin != nullptr && rope_q && q == nullptr)
        return PKV_ERR_INVALID_ARG;
    if (rope_cos_sin != nullptr && (rope_max_pos <= 0 || !aligned(rope_cos_sin, 16)))
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) ||
        !aligned(v_pool, 16) || (q != nullptr && !aligned(q, 16)) || !aligned(kv_indptr, 4) ||
        !aligned(seq_lens, 4) || (kv_indices != nullptr && !aligned(kv_indices, 4)) ||
        (status != nullptr && !aligned(status, 4)))
        return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

pkv_status launch_append(const pkv_dims *dims, void *q, const void *k_new, const void *v_new,
                         void *k_pool, void *v_pool, const int32_t *kv_indices,
                         const int32_t *kv_indptr, const int32_t *seq_lens,
                         const float *rope_cos_sin, int rope_max_pos, int rope_q,
                         uint32_t *status, pkv_stream_t stream)
{
    pkv::AppendParams p{};
    p.q = static_cast<__nv_bfloat16 *>(q);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.k_pool = static_cast<__nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<__nv_bfloat16 *>(v_pool);
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.seq_lens = seq_lens;
    p.rope = rope_cos_sin;
    p.status = status;
    p.B = dims->B;
    p.Hq = dims->Hq;
    p.Hkv = dims->Hkv;
    p.D = dims->D;
    p.page_size = dims->page_size;
    p.num_pages = dims->num_pages;
    p.num_indices = dims->num_indices;
    p.max_seq_len = dims->max_seq_len;
    p.rope_max_pos = rope_max_pos;
    p.rope_q = rope_q ? 1 : 0;
    return launch_status(pkv::launch_append(p, (cudaStream_t)stream));
}

pkv_status check_advance_args(const pkv_dims *dims, const int32_t *seq_lens,
                              const int32_t *kv_indptr, const int32_t *kv_indices,
                              const int32_t *free_pages, int num_free, const int32_t *free_head,
                              const uint32_t *status)
{
    if (seq_lens == nullptr || kv_indptr == nullptr || free_head == nullptr || num_free < 0 ||
        (num_free > 0 && free_pages == nullptr) ||
        (dims->num_indices > 0 && kv_indices == nullptr))
        return PKV_ERR_INVALID_ARG;
    if (!aligned(seq_lens, 4) || !aligned(kv_indptr, 4) || !aligned(free_head, 4) ||
        (kv_indices != nullptr && !aligned(kv_indices, 4)) ||
        (free_pages != nullptr && !aligned(free_pages, 4)) ||
        (status != nullptr && !aligned(status, 4)))
        return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

pkv::AdvanceParams advance_params(const pkv_dims *dims, int32_t *seq_lens,
                                  const int32_t *kv_indptr, int32_t *kv_indices,
                                  const int32_t *free_pages, int num_free, int32_t *free_head,
                                  uint32_t *status)
{
    pkv::AdvanceParams p{};
    p.seq_lens = seq_lens;
    p.kv_indptr = kv_indptr;
    p.kv_indices = kv_indices;
    p.free_pages = free_pages;
    p.free_head = free_head;
    p.status = status;
    p.B = dims->B;
    p.page_size = dims->page_size;
    p.max_seq_len = dims->max_seq_len;
    p.num_indices = dims->num_indices;
    p.num_free = num_free;
    return p;
}

} // namespace

extern "C" pkv_status paged_kv_extend(const pkv_dims *dims, void *q, const void *k_new,
                                      const void *v_new, const int32_t *qo_indptr, int total_q,
                                      void *k_pool, void *v_pool, const int32_t *kv_indices,
                                      const int32_t *kv_indptr, const int32_t *seq_lens,
                                      const float *rope_cos_sin, int rope_max_pos, int rope_q,
                                      uint32_t *status, pkv_stream_t stream)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (total_q < 0)
        return PKV_ERR_INVALID_ARG;
    if (dims->B == 0 || total_q == 0)
        return PKV_OK;
    if (qo_indptr == nullptr || !aligned(qo_indptr, 4))
        return PKV_ERR_INVALID_ARG;
    // the same checks as the one-token append (q, pools, tables, RoPE table)
    st = check_append_args(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                           seq_lens, rope_cos_sin, rope_max_pos, rope_q, status);
    if (st != PKV_OK)
        return st;
    pkv::AppendParams p{};
    p.q = static_cast<__nv_bfloat16 *>(q);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.k_pool = static_cast<__nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<__nv_bfloat16 *>(v_pool);
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.seq_lens = seq_lens;
    p.rope = rope_cos_sin;
    p.status = status;
    p.B = dims->B;
    p.Hq = dims->Hq;
    p.Hkv = dims->Hkv;
    p.D = dims->D;
    p.page_size = dims->page_size;
    p.num_pages = dims->num_pages;
    p.num_indices = dims->num_indices;
    p.max_seq_len = dims->max_seq_len;
    p.rope_max_pos = rope_max_pos;
    p.rope_q = rope_q ? 1 : 0;
    p.qo_indptr = qo_indptr;
    p.total_q = total_q;
    return launch_status(pkv::launch_extend(p, (cudaStream_t)stream));
}

extern "C" {

int pkv_version(void)
{
    return (1 << 16) | 3;
}

const char *pkv_status_str(pkv_status s)
{
    switch (s) {
    case PKV_OK:
        return "ok";
    case PKV_ERR_INVALID_ARG:
        return "invalid argument";
    case PKV_ERR_UNSUPPORTED:
        return "unsupported shape";
    case PKV_ERR_WORKSPACE_TOO_SMALL:
        return "workspace too small";
    case PKV_ERR_LAUNCH:
        return "kernel launch failed";
    }
    return "unknown status";
}

int pkv_split_chunk(const pkv_dims *dims, int num_splits)
{
    if (check_dims(dims) != PKV_OK || num_splits < 1 || num_splits > kMaxSplits)
        return 0;
    return chunk_for(dims, num_splits);
}

pkv_status pkv_workspace_layout(const pkv_dims *dims, int num_splits, size_t *ml_offset,
                                size_t *o_offset)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (num_splits < 1 || num_splits > kMaxSplits || ml_offset == nullptr ||
        o_offset == nullptr)
        return PKV_ERR_INVALID_ARG;
    const Layout L = layout_for(dims, num_splits);
    *ml_offset = L.split_ml_off;
    *o_offset = L.split_o_off;
    return PKV_OK;
}

size_t pkv_workspace_bytes(const pkv_dims *dims, int num_splits)
{
    if (check_dims(dims) != PKV_OK || num_splits < 1 || num_splits > kMaxSplits)
        return 0;
    return layout_for(dims, num_splits).total;
}

pkv_status pkv_plan(const pkv_dims *dims, int num_sms, int *num_splits, size_t *ws_bytes)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (num_sms <= 0 || num_splits == nullptr)
        return PKV_ERR_INVALID_ARG;
    long long s;
    if (fused_path_ok(dims)) {
        // one persistent block per SM, each with at least kFusedMinTokens
        const Layout L = layout_for(dims, 1);
        const long long work = (long long)(L.Bv > 0 ? L.Bv : 1) * dims->max_seq_len;
        s = (work + pkv::kFusedMinTokens - 1) / pkv::kFusedMinTokens;
        if (s > num_sms)
            s = num_sms;
    } else {
        const long long units = (long long)(dims->B > 0 ? dims->B : 1) * dims->Hkv;
        const long long slots = (long long)num_sms * pkv::split_decode_blocks_per_sm(dims->D);
        const long long target = 4 * slots;             // a few waves of blocks
        s = (target + units - 1) / units;
        long long s_max = ((long long)dims->max_seq_len + kMinChunkTokens - 1) / kMinChunkTokens;
        if (s > s_max)
            s = s_max;
    }
    if (s < 1)
        s = 1;
    *num_splits = (int)s;
    if (ws_bytes != nullptr)
        *ws_bytes = pkv_workspace_bytes(dims, (int)s);
    return PKV_OK;
}

pkv_status pkv_workspace_init(void *workspace, size_t ws_bytes, pkv_stream_t stream)
{
    if (workspace == nullptr || ws_bytes < kHeaderBytes || !aligned(workspace, 256))
        return PKV_ERR_INVALID_ARG;
    return launch_status(cudaMemsetAsync(workspace, 0, kHeaderBytes, (cudaStream_t)stream));
}

pkv_status pkv_rope_table(float *cos_sin, int max_pos, int D, double base,
                          pkv_stream_t stream)
{
    if (cos_sin == nullptr || max_pos <= 0 || D <= 0 || (D & 1) || !(base > 0.0) ||
        !std::isfinite(base) || !aligned(cos_sin, 16))
        return PKV_ERR_INVALID_ARG;
    return launch_status(pkv::launch_rope_table(cos_sin, max_pos, D, base, (cudaStream_t)stream));
}

pkv_status paged_kv_append(const pkv_dims *dims, void *q, const void *k_new, const void *v_new,
                           void *k_pool, void *v_pool, const int32_t *kv_indices,
                           const int32_t *kv_indptr, const int32_t *seq_lens,
                           const float *rope_cos_sin, int rope_max_pos, int rope_q,
                           uint32_t *status, pkv_stream_t stream)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (dims->B == 0)
        return PKV_OK;
    st = check_append_args(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                           seq_lens, rope_cos_sin, rope_max_pos, rope_q, status);
    if (st != PKV_OK)
        return st;
    return launch_append(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                         seq_lens, rope_cos_sin, rope_max_pos, rope_q, status, stream);
}

pkv_status paged_kv_advance(const pkv_dims *dims, int32_t *seq_lens, const int32_t *kv_indptr,
                            int32_t *kv_indices, const int32_t *free_pages, int num_free,
                            int32_t *free_head, uint32_t *status, pkv_stream_t stream)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (dims->B == 0)
        return PKV_OK;
    st = check_advance_args(dims, seq_lens, kv_indptr, kv_indices, free_pages, num_free,
                            free_head, status);
    if (st != PKV_OK)
        return st;
    const pkv::AdvanceParams p = advance_params(dims, seq_lens, kv_indptr, kv_indices,
                                                free_pages, num_free, free_head, status);
    return launch_status(pkv::launch_advance(p, (cudaStream_t)stream));
}

static pkv_status decode_attn_impl(const pkv_dims *dims, const void *q, const void *k_pool,
                                   const void *v_pool, const int32_t *kv_indices,
                                   const int32_t *kv_indptr, const int32_t *seq_lens,
                                   int num_splits, void *workspace, size_t ws_bytes, void *out,
                                   pkv_stream_t stream, bool planned)
{
    pkv_status st = check_decode_args(dims, q, k_pool, v_pool, kv_indices, kv_indptr,
                                      seq_lens, num_splits, workspace, ws_bytes, out, true);
    if (st != PKV_OK || dims->B == 0)
        return st;
    if (fused_path_ok(dims))
        return launch_persistent(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                                 num_splits, workspace, out, nullptr, nullptr, nullptr, 0,
                                 stream, nullptr, planned);
    const bool direct = num_splits == 1;
    st = launch_split(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, num_splits,
                      workspace, out, direct, stream);
    if (st != PKV_OK || direct)
        return st;
    return launch_combine_split(dims, num_splits, workspace, out, stream);
}

pkv_status paged_decode_attn(const pkv_dims *dims, const void *q, const void *k_pool,
                             const void *v_pool, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *seq_lens, int num_splits,
                             void *workspace, size_t ws_bytes, void *out, pkv_stream_t stream)
{
    return decode_attn_impl(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                            num_splits, workspace, ws_bytes, out, stream, false);
}

pkv_status paged_decode_attn_planned(const pkv_dims *dims, const void *q, const void *k_pool,
                                     const void *v_pool, const int32_t *kv_indices,
                                     const int32_t *kv_indptr, const int32_t *seq_lens,
                                     int num_splits, void *workspace, size_t ws_bytes,
                                     void *out, pkv_stream_t stream)
{
    return decode_attn_impl(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                            num_splits, workspace, ws_bytes, out, stream, true);
}

pkv_status paged_decode_plan(const pkv_dims *dims, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *seq_lens, int num_splits,
                             void *workspace, size_t ws_bytes, pkv_stream_t stream)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (num_splits < 1 || num_splits > kMaxSplits)
        return PKV_ERR_INVALID_ARG;
    if (dims->B == 0)
        return PKV_OK;
    if (kv_indptr == nullptr || seq_lens == nullptr || workspace == nullptr ||
        (dims->num_indices > 0 && kv_indices == nullptr) || !aligned(workspace, 256) ||
        !aligned(kv_indptr, 4) || !aligned(seq_lens, 4) ||
        (kv_indices != nullptr && !aligned(kv_indices, 4)))
        return PKV_ERR_INVALID_ARG;
    const size_t need = pkv_workspace_bytes(dims, num_splits);
    if (need == 0)
        return PKV_ERR_INVALID_ARG;
    if (ws_bytes < need)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!fused_path_ok(dims))
        return PKV_OK;                     // other shapes compute their split per call
    const Layout L = layout_for(dims, num_splits);
    char *ws = static_cast<char *>(workspace);
    const pkv::FusedParams p = persistent_params(dims, L, ws, kv_indices, kv_indptr, seq_lens);
    return launch_status(pkv::launch_decode_plan(
        p, num_splits, reinterpret_cast<int32_t *>(ws + L.plan_off), (cudaStream_t)stream));
}

static pkv_status decode_step_impl(const pkv_dims *dims, const void *q, const void *k_new,
                                   const void *v_new, void *k_pool, void *v_pool,
                                   const int32_t *kv_indices, const int32_t *kv_indptr,
                                   const int32_t *seq_lens, const float *rope_cos_sin,
                                   int rope_max_pos, int num_splits, void *workspace,
                                   size_t ws_bytes, void *out, pkv_stream_t stream, bool planned)
{
    pkv_status st = check_decode_args(dims, q, k_pool, v_pool, kv_indices, kv_indptr,
                                      seq_lens, num_splits, workspace, ws_bytes, out, true);
    if (st != PKV_OK || dims->B == 0)
        return st;
    uint32_t *status = static_cast<uint32_t *>(workspace);
    st = check_append_args(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                           seq_lens, rope_cos_sin, rope_max_pos, 0, status);
    if (st != PKV_OK)
        return st;
    if (fused_path_ok(dims))
        return launch_persistent(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                                 num_splits, workspace, out, k_new, v_new, rope_cos_sin,
                                 rope_max_pos, stream, nullptr, planned);
    // other shapes: rotate a copy of q in the workspace, append, then decode
    const Layout L = layout_for(dims, num_splits);
    void *qs = static_cast<char *>(workspace) + L.qscratch_off;
    const size_t qbytes = (size_t)dims->B * dims->Hq * dims->D * 2;
    st = launch_status(
        cudaMemcpyAsync(qs, q, qbytes, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
    if (st != PKV_OK)
        return st;
    st = launch_append(dims, qs, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                       rope_cos_sin, rope_max_pos, rope_cos_sin != nullptr, status, stream);
    if (st != PKV_OK)
        return st;
    const bool direct = num_splits == 1;
    st = launch_split(dims, qs, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, num_splits,
                      workspace, out, direct, stream);
    if (st != PKV_OK || direct)
        return st;
    return launch_combine_split(dims, num_splits, workspace, out, stream);
}

pkv_status paged_decode_step(const pkv_dims *dims, const void *q, const void *k_new,
                             const void *v_new, void *k_pool, void *v_pool,
                             const int32_t *kv_indices, const int32_t *kv_indptr,
                             const int32_t *seq_lens, const float *rope_cos_sin,
                             int rope_max_pos, int num_splits, void *workspace,
                             size_t ws_bytes, void *out, pkv_stream_t stream)
{
    return decode_step_impl(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                            seq_lens, rope_cos_sin, rope_max_pos, num_splits, workspace,
                            ws_bytes, out, stream, false);
}

pkv_status paged_decode_step_planned(const pkv_dims *dims, const void *q, const void *k_new,
                                     const void *v_new, void *k_pool, void *v_pool,
                                     const int32_t *kv_indices, const int32_t *kv_indptr,
                                     const int32_t *seq_lens, const float *rope_cos_sin,
                                     int rope_max_pos, int num_splits, void *workspace,
                                     size_t ws_bytes, void *out, pkv_stream_t stream)
{
    return decode_step_impl(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                            seq_lens, rope_cos_sin, rope_max_pos, num_splits, workspace,
                            ws_bytes, out, stream, true);
}

pkv_status paged_decode_step_advance(const pkv_dims *dims, const void *q, const void *k_new,
                                     const void *v_new, void *k_pool, void *v_pool,
                                     int32_t *kv_indices, const int32_t *kv_indptr,
                                     int32_t *seq_lens, const float *rope_cos_sin,
                                     int rope_max_pos, int num_splits, void *workspace,
                                     size_t ws_bytes, void *out, const int32_t *free_pages,
                                     int num_free, int32_t *free_head, pkv_stream_t stream)
{
    pkv_status st = check_decode_args(dims, q, k_pool, v_pool, kv_indices, kv_indptr,
                                      seq_lens, num_splits, workspace, ws_bytes, out, true);
    if (st != PKV_OK || dims->B == 0)
        return st;
    uint32_t *status = static_cast<uint32_t *>(workspace);
    st = check_append_args(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                           seq_lens, rope_cos_sin, rope_max_pos, 0, status);
    if (st != PKV_OK)
        return st;
    st = check_advance_args(dims, seq_lens, kv_indptr, kv_indices, free_pages, num_free,
                            free_head, status);
    if (st != PKV_OK)
        return st;
    const pkv::AdvanceParams adv = advance_params(dims, seq_lens, kv_indptr, kv_indices,
                                                  free_pages, num_free, free_head, status);
    // The piece combine runs after the decode grid has completed and never
    // reads the metadata, so one extra block of it can advance that metadata.
    if (fused_path_ok(dims) && num_splits > 1)
        return launch_persistent(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                                 num_splits, workspace, out, k_new, v_new, rope_cos_sin,
                                 rope_max_pos, stream, &adv);
    st = paged_decode_step(dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                           seq_lens, rope_cos_sin, rope_max_pos, num_splits, workspace,
                           ws_bytes, out, stream);
    if (st != PKV_OK)
        return st;
    return launch_status(pkv::launch_advance(adv, (cudaStream_t)stream));
}

static pkv_status contig_impl(const pkv_dims *dims, const void *q, const void *k_new,
                              const void *v_new, void *k_cache, void *v_cache,
                              const int32_t *cache_batch_idx, const int32_t *seq_lens,
                              const float *rope_cos_sin, int rope_max_pos, int num_splits,
                              void *workspace, size_t ws_bytes, void *out, pkv_stream_t stream,
                              bool planned)
{
    if (dims == nullptr)
        return PKV_ERR_INVALID_ARG;
    pkv_dims d = *dims;
    d.num_indices = d.B;                       // one table entry per row
    pkv_status st = check_dims(&d);
    if (st != PKV_OK)
        return st;
    if (d.B == 0)
        return PKV_OK;
    if ((k_new == nullptr) != (v_new == nullptr) || workspace == nullptr ||
        !aligned(workspace, 256) ||
        (cache_batch_idx != nullptr && !aligned(cache_batch_idx, 4)))
        return PKV_ERR_INVALID_ARG;
    if (num_splits < 1 || num_splits > kMaxSplits)
        return PKV_ERR_INVALID_ARG;
    const size_t need = pkv_workspace_bytes(&d, num_splits);
    if (need == 0)
        return PKV_ERR_INVALID_ARG;
    if (ws_bytes < need)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    const Layout L = layout_for(&d, num_splits);
    int32_t *kv_indptr = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + L.table_off);
    int32_t *kv_indices = kv_indptr + d.B + 1;
    // a planned call finds the table, like the plan, where the step's first
    // call left it
    if (!planned) {
        st = launch_status(
            pkv::launch_contig_table(cache_batch_idx, d.B, kv_indptr, (cudaStream_t)stream));
        if (st != PKV_OK)
            return st;
    }
    if (k_new != nullptr)
        return decode_step_impl(&d, q, k_new, v_new, k_cache, v_cache, kv_indices, kv_indptr,
                                seq_lens, rope_cos_sin, rope_max_pos, num_splits, workspace,
                                ws_bytes, out, stream, planned);
    return decode_attn_impl(&d, q, k_cache, v_cache, kv_indices, kv_indptr, seq_lens,
                            num_splits, workspace, ws_bytes, out, stream, planned);
}

pkv_status decode_attn_contig(const pkv_dims *dims, const void *q, const void *k_new,
                              const void *v_new, void *k_cache, void *v_cache,
                              const int32_t *cache_batch_idx, const int32_t *seq_lens,
                              const float *rope_cos_sin, int rope_max_pos, int num_splits,
                              void *workspace, size_t ws_bytes, void *out, pkv_stream_t stream)
{
    return contig_impl(dims, q, k_new, v_new, k_cache, v_cache, cache_batch_idx, seq_lens,
                       rope_cos_sin, rope_max_pos, num_splits, workspace, ws_bytes, out, stream,
                       false);
}

pkv_status decode_attn_contig_planned(const pkv_dims *dims, const void *q, const void *k_new,
                                      const void *v_new, void *k_cache, void *v_cache,
                                      const int32_t *cache_batch_idx, const int32_t *seq_lens,
                                      const float *rope_cos_sin, int rope_max_pos,
                                      int num_splits, void *workspace, size_t ws_bytes,
                                      void *out, pkv_stream_t stream)
{
    return contig_impl(dims, q, k_new, v_new, k_cache, v_cache, cache_batch_idx, seq_lens,
                       rope_cos_sin, rope_max_pos, num_splits, workspace, ws_bytes, out, stream,
                       true);
}

pkv_status pkv_prefill_plan(const pkv_dims *dims, int max_q_len, int num_sms, size_t ws_bytes,
                            int32_t *plan)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (plan == nullptr || max_q_len < 0 || num_sms < 1 || num_sms > pkv::kPrefillMaxSms)
        return PKV_ERR_INVALID_ARG;
    pkv::PrefillPlan pl;
    const int n_rep = dims->Hq / dims->Hkv;
    if (!pkv::prefill_plan(dims->B, dims->Hkv, 128 / n_rep, max_q_len, num_sms, dims->D,
                           ws_bytes, &pl))
        return PKV_ERR_UNSUPPORTED;
    const int32_t v[7] = {pl.pairs, pl.units, pl.group_rows, pl.entries, pl.split,
                          pl.split_base, pl.grid};
    for (int i = 0; i < 7; ++i)
        plan[i] = v[i];
    return PKV_OK;
}

size_t pkv_prefill_workspace_bytes(int D, int num_sms)
{
    if ((D != 64 && D != 128) || num_sms <= 0 || num_sms > pkv::kPrefillMaxSms)
        return 0;
    return (size_t)num_sms * pkv::prefill_slot_bytes(D);
}

namespace {

pkv_status prefill_impl(const pkv_dims *dims, const void *q, const int32_t *qo_indptr,
                        int total_q, int max_q_len, const void *k_pool, const void *v_pool,
                        const int32_t *kv_indices, const int32_t *kv_indptr,
                        const int32_t *seq_lens, void *workspace, size_t ws_bytes, void *out,
                        uint32_t *status, pkv_stream_t stream)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (total_q < 0 || max_q_len < 0 || !(dims->scale > 0.f))
        return PKV_ERR_INVALID_ARG;
    if (workspace != nullptr && !aligned(workspace, 256))
        return PKV_ERR_INVALID_ARG;
    if (dims->B == 0 || total_q == 0 || max_q_len == 0)
        return PKV_OK;
    if ((long long)dims->B * dims->Hkv > 65535)
        return PKV_ERR_UNSUPPORTED;
    // the kernel keeps pool offsets in 16-byte units as 32-bit integers
    if ((double)dims->num_pages * dims->page_size * dims->Hkv * dims->D / 8 >= 4294967295.0)
        return PKV_ERR_UNSUPPORTED;
    if (q == nullptr || qo_indptr == nullptr || k_pool == nullptr || v_pool == nullptr ||
        kv_indptr == nullptr || seq_lens == nullptr || out == nullptr ||
        (dims->num_indices > 0 && kv_indices == nullptr))
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(qo_indptr, 4) || !aligned(kv_indptr, 4) || !aligned(seq_lens, 4) ||
        (kv_indices != nullptr && !aligned(kv_indices, 4)) ||
        (status != nullptr && !aligned(status, 4)))
        return PKV_ERR_INVALID_ARG;
    pkv::PrefillParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.qo_indptr = qo_indptr;
    p.k_pool = static_cast<const __nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16 *>(v_pool);
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.seq_lens = seq_lens;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.status = status;
    p.B = dims->B;
    p.Hq = dims->Hq;
    p.Hkv = dims->Hkv;
    p.n_rep = dims->Hq / dims->Hkv;
    p.page_size = dims->page_size;
    p.ps_shift = log2_exact(dims->page_size);
    p.num_pages = dims->num_pages;
    p.num_indices = dims->num_indices;
    p.max_seq_len = dims->max_seq_len;
    p.total_q = total_q;
    p.tq = 128 / p.n_rep;
    p.scale_log2 = (float)((double)dims->scale * 1.4426950408889634);
    return launch_status(pkv::launch_prefill(p, dims->D, max_q_len, workspace,
                                             workspace != nullptr ? ws_bytes : 0,
                                             (cudaStream_t)stream));
}

} // namespace

pkv_status paged_prefill_attn(const pkv_dims *dims, const void *q, const int32_t *qo_indptr,
                              int total_q, int max_q_len, const void *k_pool, const void *v_pool,
                              const int32_t *kv_indices, const int32_t *kv_indptr,
                              const int32_t *seq_lens, void *out, uint32_t *status,
                              pkv_stream_t stream)
{
    return prefill_impl(dims, q, qo_indptr, total_q, max_q_len, k_pool, v_pool, kv_indices,
                        kv_indptr, seq_lens, nullptr, 0, out, status, stream);
}

pkv_status paged_prefill_attn_ws(const pkv_dims *dims, const void *q, const int32_t *qo_indptr,
                                 int total_q, int max_q_len, const void *k_pool,
                                 const void *v_pool, const int32_t *kv_indices,
                                 const int32_t *kv_indptr, const int32_t *seq_lens,
                                 void *workspace, size_t ws_bytes, void *out, uint32_t *status,
                                 pkv_stream_t stream)
{
    return prefill_impl(dims, q, qo_indptr, total_q, max_q_len, k_pool, v_pool, kv_indices,
                        kv_indptr, seq_lens, workspace, ws_bytes, out, status, stream);
}

pkv_status paged_decode_partials(const pkv_dims *dims, const void *q, const void *k_pool,
                                 const void *v_pool, const int32_t *kv_indices,
                                 const int32_t *kv_indptr, const int32_t *seq_lens,
                                 int num_splits, void *workspace, size_t ws_bytes,
                                 pkv_stream_t stream)
{
    pkv_status st = check_decode_args(dims, q, k_pool, v_pool, kv_indices, kv_indptr,
                                      seq_lens, num_splits, workspace, ws_bytes, nullptr, false);
    if (st != PKV_OK || dims->B == 0)
        return st;
    return launch_split(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, num_splits,
                        workspace, nullptr, false, stream);
}

pkv_status decode_combine(const pkv_dims *dims, const float *o_part, const float *ml_part,
                          int num_splits, void *out, pkv_stream_t stream)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (num_splits < 1 || num_splits > kMaxSplits)
        return PKV_ERR_INVALID_ARG;
    if (dims->B == 0)
        return PKV_OK;
    if (o_part == nullptr || ml_part == nullptr || out == nullptr || !aligned(o_part, 16) ||
        !aligned(ml_part, 8) || !aligned(out, 16))
        return PKV_ERR_INVALID_ARG;
    pkv::CombineParams p{};
    p.o_part = o_part;
    p.ml_part = ml_part;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.B = dims->B;
    p.Hq = dims->Hq;
    p.D = dims->D;
    p.num_splits = num_splits;
    return launch_status(pkv::launch_combine(p, (cudaStream_t)stream));
}

} // extern "C"
