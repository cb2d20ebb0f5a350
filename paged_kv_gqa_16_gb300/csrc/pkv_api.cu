// pkv_api.cu -- the C ABI of libpkv (declared in include/pkv.h): argument
// checks, the split planner, the workspace layout and kernel dispatch.
// Nothing here allocates, synchronises or prints.
#include <cmath>
#include <cstdint>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kHeaderBytes = 256;
constexpr int kMaxSplits = 65536;
constexpr int kMinChunkTokens = 256;   // the planner does not split finer than this

size_t round_up(size_t x, size_t a)
{
    return (x + a - 1) / a * a;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Shape checks common to every entry point.
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

pkv_status launch_status(cudaError_t e)
{
    return e == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

pkv_status decode_common(const pkv_dims *dims, const void *q, const void *k_pool,
                         const void *v_pool, const int32_t *kv_indices,
                         const int32_t *kv_indptr, const int32_t *seq_lens, int num_splits,
                         void *workspace, size_t ws_bytes, void *out, bool direct,
                         pkv_stream_t stream)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (num_splits < 1 || num_splits > kMaxSplits)
        return PKV_ERR_INVALID_ARG;
    if (dims->B == 0)
        return PKV_OK;
    if (q == nullptr || k_pool == nullptr || v_pool == nullptr || kv_indptr == nullptr ||
        seq_lens == nullptr || workspace == nullptr || (direct && out == nullptr))
        return PKV_ERR_INVALID_ARG;
    if (dims->num_indices > 0 && kv_indices == nullptr)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(workspace, 256) || (direct && !aligned(out, 16)) ||
        !aligned(kv_indptr, 4) || !aligned(seq_lens, 4) ||
        (kv_indices != nullptr && !aligned(kv_indices, 4)))
        return PKV_ERR_INVALID_ARG;
    const size_t need = pkv_workspace_bytes(dims, num_splits);
    if (need == 0)
        return PKV_ERR_INVALID_ARG;
    if (ws_bytes < need)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    size_t ml_off = 0, o_off = 0;
    pkv_workspace_layout(dims, num_splits, &ml_off, &o_off);

    pkv::DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_pool = static_cast<const __nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16 *>(v_pool);
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.seq_lens = seq_lens;
    p.ml_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + ml_off);
    p.o_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_off);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.status = static_cast<uint32_t *>(workspace);
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

} // namespace

extern "C" {

int pkv_version(void)
{
    return (1 << 16) | 0;
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
    const size_t rows = (size_t)dims->B * dims->Hq * num_splits;
    *ml_offset = kHeaderBytes;
    *o_offset = kHeaderBytes + round_up(rows * 2 * sizeof(float), 256);
    return PKV_OK;
}

size_t pkv_workspace_bytes(const pkv_dims *dims, int num_splits)
{
    size_t ml = 0, o = 0;
    if (pkv_workspace_layout(dims, num_splits, &ml, &o) != PKV_OK)
        return 0;
    const size_t rows = (size_t)dims->B * dims->Hq * num_splits;
    return o + round_up(rows * dims->D * sizeof(float), 256);
}

pkv_status pkv_plan(const pkv_dims *dims, int num_sms, int *num_splits, size_t *ws_bytes)
{
    pkv_status st = check_dims(dims);
    if (st != PKV_OK)
        return st;
    if (num_sms <= 0 || num_splits == nullptr)
        return PKV_ERR_INVALID_ARG;
    const long long units = (long long)(dims->B > 0 ? dims->B : 1) * dims->Hkv;
    const long long slots = (long long)num_sms * pkv::split_decode_blocks_per_sm(dims->D);
    const long long target = 4 * slots;             // a few waves of blocks
    long long s = (target + units - 1) / units;
    long long s_max = ((long long)dims->max_seq_len + kMinChunkTokens - 1) / kMinChunkTokens;
    if (s_max < 1)
        s_max = 1;
    if (s > s_max)
        s = s_max;
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

pkv_status paged_decode_attn(const pkv_dims *dims, const void *q, const void *k_pool,
                             const void *v_pool, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *seq_lens, int num_splits,
                             void *workspace, size_t ws_bytes, void *out, pkv_stream_t stream)
{
    if (out == nullptr && dims != nullptr && dims->B > 0)
        return PKV_ERR_INVALID_ARG;
    const bool direct = num_splits == 1;
    pkv_status st = decode_common(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                                  num_splits, workspace, ws_bytes, out, direct, stream);
    if (st != PKV_OK || direct || dims->B == 0)
        return st;
    size_t ml_off = 0, o_off = 0;
    pkv_workspace_layout(dims, num_splits, &ml_off, &o_off);
    return decode_combine(dims,
                          reinterpret_cast<const float *>(static_cast<char *>(workspace) + o_off),
                          reinterpret_cast<const float *>(static_cast<char *>(workspace) + ml_off),
                          num_splits, out, stream);
}

pkv_status paged_decode_partials(const pkv_dims *dims, const void *q, const void *k_pool,
                                 const void *v_pool, const int32_t *kv_indices,
                                 const int32_t *kv_indptr, const int32_t *seq_lens,
                                 int num_splits, void *workspace, size_t ws_bytes,
                                 pkv_stream_t stream)
{
    return decode_common(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, num_splits,
                         workspace, ws_bytes, nullptr, false, stream);
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
