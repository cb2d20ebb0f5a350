// pkv_append.cu -- kernel (1): fused RoPE + K/V append into a paged pool,
// and the set-up kernel that fills the RoPE cos/sin table.
//
// What it computes (AstrAI commit log): the decode step writes the new
// token's K/V at its slot before attending (compare v1.3.12..6f09b1d,
// astrai/extension/attention_backend.py, CudaBackend.fwd_decode writing
// k_buffer[layer, out_cache_loc]); the slot of position pos is
// page_table[pos / page_size] * page_size + pos % page_size (cache.py,
// PagePool._extend_slot) and the position is seq_len - 1 (cache.py,
// bind_tasks).  K is rotated first (commits by author: "extend CUDA rotary
// embedding to packed 3d inputs", "cos/sin freqs_cis table"): each
// interleaved pair is multiplied by the unit complex number (cos, sin) of
// pos * theta_i.
//
// Layout of the work: one block per row (append) or per new token (extend);
// each thread moves 16-byte vectors (8 bf16 = 4 rotation pairs) of the
// token's Hkv K/V head vectors and, when asked, its Hq query heads.  The page
// lookup happens once per block.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

// One token: row b, position pos; its K/V (and, with rope_q, its query
// heads) are input row t of k_new / v_new / q.  Page lookup, checks, K
// rotated by pos, V copied, both stored at the token's slot.
__device__ __forceinline__ void write_token(const AppendParams &p, int b, int pos, size_t t)
{
    const int pg0 = p.kv_indptr[b], pg1 = p.kv_indptr[b + 1];
    unsigned bad = 0;
    int page = 0;
    const int pi = pos / p.page_size;
    if (pg0 < 0 || pg1 < pg0 || pg1 > p.num_indices || pi >= pg1 - pg0) {
        bad |= kFlagBadPage;
    } else {
        page = p.kv_indices[pg0 + pi];
        if (page < 0 || page >= p.num_pages)
            bad |= kFlagBadPage;
    }
    if (p.rope != nullptr && pos >= p.rope_max_pos)
        bad |= kFlagBadPos;
    if (bad) {
        if (p.status != nullptr && threadIdx.x == 0)
            atomicOr(p.status, bad);
        return;
    }
    const int slot = pos - pi * p.page_size;
    const int D = p.D;
    const int vpr = D >> 3;  // 16-byte vectors per head vector
    const size_t row_off = ((size_t)page * p.page_size + slot) * (size_t)p.Hkv * D;
    const float *cs = p.rope != nullptr ? p.rope + (size_t)pos * D : nullptr;

    const uint4 *kin = reinterpret_cast<const uint4 *>(p.k_new + t * p.Hkv * D);
    const uint4 *vin = reinterpret_cast<const uint4 *>(p.v_new + t * p.Hkv * D);
    uint4 *kout = reinterpret_cast<uint4 *>(p.k_pool + row_off);
    uint4 *vout = reinterpret_cast<uint4 *>(p.v_pool + row_off);
    for (int it = threadIdx.x; it < p.Hkv * vpr; it += blockDim.x) {
        const int c = it % vpr;
        uint4 k = kin[it];
        if (cs != nullptr) {
            const float4 *c4 = reinterpret_cast<const float4 *>(cs + 8 * c);
            k = rotate_pairs8(k, c4[0], c4[1]);
        }
        kout[it] = k;
        vout[it] = vin[it];
    }
    if (cs != nullptr && p.rope_q) {
        uint4 *qrow = reinterpret_cast<uint4 *>(p.q + t * p.Hq * D);
        for (int it = threadIdx.x; it < p.Hq * vpr; it += blockDim.x) {
            const int c = it % vpr;
            const float4 *c4 = reinterpret_cast<const float4 *>(cs + 8 * c);
            qrow[it] = rotate_pairs8(qrow[it], c4[0], c4[1]);
        }
    }
}

__global__ void __launch_bounds__(128) append_kernel(const AppendParams p)
{
    // the decode launched next may start its prologue; it waits for this
    // grid's completion before it reads q or the pools
    grid_launch_dependents();
    const int b = blockIdx.x;
    const int L = p.seq_lens[b];
    if (L <= 0) {
        if (L < 0 && p.status != nullptr && threadIdx.x == 0)
            atomicOr(p.status, kFlagBadLen);
        return;
    }
    write_token(p, b, L - 1, (size_t)b);
}

// Extend: one block per new token t of the flattened chunks.  Its row is the
// last b with qo_indptr[b] <= t; row b's chunk is the last q_len of its L
// tokens, so token t sits at position L - q_len + (t - qo_indptr[b]).
__global__ void __launch_bounds__(128) extend_kernel(const AppendParams p)
{
    grid_launch_dependents();
    const int t = blockIdx.x;
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.qo_indptr[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int b = lo;
    const int a = p.qo_indptr[b], e = p.qo_indptr[b + 1];
    const int L = p.seq_lens[b];
    const int q_len = e - a;
    if (t < a || t >= e || q_len > L || L > p.max_seq_len) {
        if (p.status != nullptr && threadIdx.x == 0)
            atomicOr(p.status, kFlagBadLen);
        return;
    }
    write_token(p, b, L - q_len + (t - a), (size_t)t);
}

// (cos, sin) of pos * base^(-2i/D), in double, rounded once to fp32.
__global__ void rope_table_kernel(float *cos_sin, int max_pos, int half, double base, int D)
{
    const long long n = (long long)max_pos * half;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
         idx += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(idx % half);
        const long long pos = idx / half;
        const double theta = pow(base, -2.0 * (double)i / (double)D);
        double s, c;
        sincos((double)pos * theta, &s, &c);
        cos_sin[2 * idx] = (float)c;
        cos_sin[2 * idx + 1] = (float)s;
    }
}

} // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream)
{
    append_kernel<<<p.B, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_extend(const AppendParams &p, cudaStream_t stream)
{
    if (p.total_q <= 0)
        return cudaSuccess;
    extend_kernel<<<p.total_q, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rope_table(float *cos_sin, int max_pos, int D, double base,
                              cudaStream_t stream)
{
    const long long n = (long long)max_pos * (D / 2);
    const int threads = 256;
    long long blocks = (n + threads - 1) / threads;
    if (blocks > 4096)
        blocks = 4096;
    if (blocks < 1)
        blocks = 1;
    rope_table_kernel<<<(int)blocks, threads, 0, stream>>>(cos_sin, max_pos, D / 2, base, D);
    return cudaGetLastError();
}

} // namespace pkv
