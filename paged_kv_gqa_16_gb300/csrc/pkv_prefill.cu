// pkv_prefill.cu -- paged ragged prefill / extend attention.
//
// What it computes (AstrAI commit log, compare v1.3.12..6f09b1d,
// astrai/extension/attention_ops.py, attn_paged_prefill and attn_prefill):
// a ragged batch of query chunks, flattened to q [total_q, Hq, D] with
// qo_indptr the prefix sum of the chunk lengths.  Row b's chunk is the last
// q_len of its L = seq_lens[b] tokens (their K/V are already in the pool), so
// query i sits at position L - q_len + i and attends, causally, keys
// 0 .. that position: out = softmax(scale q K^T) V with K/V of kv head
// h / n_rep gathered through the page table.
//
// Layout of the work.  A block takes one (row, kv head, tile of query
// tokens); its 64 query rows are the tile's tokens x the kv head's n_rep
// query heads (token-major), so the tile holds 64 / n_rep tokens.  Per key
// tile of 64 tokens:
//  - a producer warp gathers the K and V rows of that kv head with 1-D bulk
//    copies (one D*2-byte row per token, looked up through the page table)
//    into a two-stage ring of padded rows (ldmatrix reads are bank-conflict
//    free), handed over by full/empty mbarriers, every wait time-bounded;
//  - four consumer warps, 16 query rows each, form S = q K^T with m16n8k16
//    bf16 tensor-core products, mask keys past each row's position, update
//    an fp32 online softmax (log2 domain), round P to bf16 and add P V.
// Key tiles entirely at or before the tile's first position need no mask.
// Row b's query tiles are handed out last tile first, so the blocks with the
// most keys start first.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr unsigned kAll = 0xffffffffu;

__device__ __forceinline__ void flag(uint32_t *status, unsigned bits)
{
    if (status != nullptr)
        atomicOr(status, bits);
}

template <int D>
struct PrefillCfg {
    static constexpr int kRows = 64;                  // query rows per block
    static constexpr int kKeys = 64;                  // keys per tile
    static constexpr int kStages = 2;
    static constexpr int kConsumers = 4;
    static constexpr int kThreads = (kConsumers + 1) * 32;
    static constexpr int kRowBytes = D * 2;
    static constexpr int kPitch = kRowBytes + 16;
    static constexpr int kQBytes = kRows * kRowBytes;
    static constexpr int kTileBytes = kKeys * kPitch;
    static constexpr int kStageBytes = 2 * kTileBytes;   // K rows, then V rows
    static constexpr int kRingOffset = kQBytes;
    static constexpr int kBarOffset = kRingOffset + kStages * kStageBytes;
    static constexpr int kPrefixOffset = kBarOffset + (2 * kStages + 1) * 8 + 8;
    static constexpr int kSmemBytes = kPrefixOffset + (kPrefillMaxRows + 1) * 4;
    static_assert(kRingOffset % 16 == 0 && kBarOffset % 8 == 0 && kPitch % 16 == 0,
                  "bulk-copy destinations need 16-byte alignment");
};

template <int D>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 2)
    prefill_kernel(const PrefillParams p)
{
    using C = PrefillCfg<D>;
    constexpr int NST = C::kStages;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *s_q = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);
    uint64_t *empty = full + NST;
    uint64_t *qbar = empty + NST;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(qbar + 1);
    int *prefix = reinterpret_cast<int *>(smem + C::kPrefixOffset);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y;                         // kv head
    const int n_rep = p.n_rep, tq = p.tq;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 32);
            mbar_init(&empty[i], C::kConsumers);
        }
        mbar_init(qbar, 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    grid_dependency_wait();

    // ---- query tiles per row, checked, then their prefix sums -------------
    for (int r = threadIdx.x; r < p.B; r += blockDim.x) {
        const int a = p.qo_indptr[r], e = p.qo_indptr[r + 1];
        const int L = p.seq_lens[r];
        int n = e - a;
        if (n < 0 || a < 0 || e > p.total_q || L < 0 || L > p.max_seq_len || n > L) {
            if (blockIdx.x == 0 && g == 0)
                flag(p.status, kFlagBadLen);
            n = 0;
        }
        prefix[r + 1] = (n + tq - 1) / tq;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int i = base + lane;
            int v = i < p.B ? prefix[i + 1] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int t = __shfl_up_sync(kAll, v, off);
                if (lane >= off)
                    v += t;
            }
            v += carry;
            if (i < p.B)
                prefix[i + 1] = v;
            carry = __shfl_sync(kAll, v, 31);
        }
        if (lane == 0)
            prefix[0] = 0;
    }
    __syncthreads();
    const int tile_id = blockIdx.x;
    if (tile_id >= prefix[p.B])
        return;
    int b = 0;
    {
        int lo = 0, hi = p.B - 1;                 // last row with prefix[row] <= tile_id
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= tile_id)
                lo = mid;
            else
                hi = mid - 1;
        }
        b = lo;
    }
    const int n_tiles = prefix[b + 1] - prefix[b];
    const int t = n_tiles - 1 - (tile_id - prefix[b]);   // last tile first
    const int q0 = p.qo_indptr[b];
    const int q_len = p.qo_indptr[b + 1] - q0;
    const int L = p.seq_lens[b];
    const int i0 = t * tq;                               // first token of the tile
    const int ntok = min(tq, q_len - i0);
    const int pos_first = L - q_len + i0;
    const int kv_end = pos_first + ntok;                 // keys [0, kv_end)
    const int n_kt = (kv_end + C::kKeys - 1) / C::kKeys;
    const int pg0 = p.kv_indptr[b];
    const int npg = p.kv_indptr[b + 1] - pg0;
    const bool table_ok = pg0 >= 0 && npg >= 0 && p.kv_indptr[b + 1] <= p.num_indices &&
                          (long long)npg * p.page_size >= (long long)L;

    if (warp == C::kConsumers) {
        // ======================= producer warp ============================
        if (!table_ok) {
            if (lane == 0)
                flag(p.status, kFlagBadPage);
        }
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(ntok * n_rep * C::kRowBytes);
            mbar_arrive_expect_tx(qbar, bytes);
            for (int i = 0; i < ntok; ++i)
                bulk_copy_g2s(s_q + (size_t)i * n_rep * C::kRowBytes,
                              p.q + ((size_t)(q0 + i0 + i) * p.Hq + (size_t)g * n_rep) * D,
                              (uint32_t)(n_rep * C::kRowBytes), qbar);
        }
        int kt = 0;
        for (; kt < n_kt; ++kt) {
            const int st = kt % NST;
            if (kt >= NST) {
                const bool ok = mbar_wait_bounded(&empty[st], (uint32_t)(((kt / NST) - 1) & 1));
                if (!__all_sync(kAll, ok) || *abort_flag) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        flag(p.status, kFlagTimeout);
                    }
                    break;
                }
            }
            fence_proxy_async_smem();
            const int tok0 = kt * C::kKeys;
            const int nvalid = min(C::kKeys, kv_end - tok0);
            unsigned char *krows = smem + C::kRingOffset + st * C::kStageBytes;
            unsigned char *vrows = krows + C::kTileBytes;
            // V rows past the last key must be finite (P is 0 there)
            for (int j = nvalid; j < C::kKeys; ++j) {
                uint4 *z = reinterpret_cast<uint4 *>(vrows + j * C::kPitch);
                for (int k = lane; k < C::kRowBytes / 16; k += 32)
                    z[k] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (lane == 0)
                mbar_arrive_expect_tx(&full[st], (uint32_t)(nvalid * 2 * C::kRowBytes));
            else
                mbar_arrive(&full[st]);
            for (int j = lane; j < nvalid; j += 32) {
                const int tok = tok0 + j;
                const int pi = p.ps_shift >= 0 ? (tok >> p.ps_shift) : (tok / p.page_size);
                const int sl = tok - pi * p.page_size;
                int page = table_ok ? __ldg(p.kv_indices + pg0 + pi) : 0;
                if (page < 0 || page >= p.num_pages) {
                    flag(p.status, kFlagBadPage);
                    page = 0;
                }
                const size_t off = (((size_t)page * p.page_size + sl) * p.Hkv + g) * D;
                bulk_copy_g2s(krows + j * C::kPitch, p.k_pool + off, C::kRowBytes, &full[st]);
                bulk_copy_g2s(vrows + j * C::kPitch, p.v_pool + off, C::kRowBytes, &full[st]);
            }
        }
        // let the copies already issued land before the block exits
        for (int k = (kt > NST ? kt - NST : 0); k < kt; ++k)
            (void)mbar_wait_bounded(&full[k % NST], (uint32_t)((k / NST) & 1));
        (void)mbar_wait_bounded(qbar, 0u);
        return;
    }

    // ========================= consumer warps ===============================
    const int fr = lane >> 2, cq = (lane & 3) * 2;
    const int k_tok = (lane & 7) + ((lane >> 4) << 3);
    const int k_col = ((lane >> 3) & 1) * 8;
    const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_col = (lane >> 4) * 8;
    const uint32_t ring_s = smem_addr(smem + C::kRingOffset);
    // this thread's two query rows (fragment rows fr and fr + 8)
    const int rows_used = tq * n_rep;
    int rr[2], pos[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        rr[h] = warp * 16 + fr + 8 * h;
        const int tok = rr[h] / n_rep;
        pos[h] = (rr[h] < rows_used && tok < ntok) ? pos_first + tok : -1;
    }
    bool aborted = false;
    {
        const bool ok = mbar_wait_bounded(qbar, 0u);
        if (!__all_sync(kAll, ok)) {
            aborted = true;
            if (lane == 0) {
                *abort_flag = 1;
                flag(p.status, kFlagTimeout);
            }
        }
    }
    uint32_t qf[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t *qr = reinterpret_cast<const uint32_t *>(s_q + rr[h] * C::kRowBytes);
            const bool live = pos[h] >= 0;
            qf[kk][h] = live ? qr[(kk * 16 + cq) / 2] : 0u;
            qf[kk][2 + h] = live ? qr[(kk * 16 + 8 + cq) / 2] : 0u;
        }
    }
    const int pos_min_block = pos_first;   // rows of this block: positions >= pos_first

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float oacc[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
        oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

    for (int kt = 0; kt < n_kt; ++kt) {
        const int st = kt % NST;
        if (!aborted) {
            const bool ok = mbar_wait_bounded(&full[st], (uint32_t)((kt / NST) & 1));
            if (!__all_sync(kAll, ok) || *abort_flag) {
                aborted = true;
                if (lane == 0) {
                    *abort_flag = 1;
                    flag(p.status, kFlagTimeout);
                }
            }
        }
        if (aborted)
            break;
        const int tok0 = kt * C::kKeys;
        const uint32_t kbase = ring_s + st * C::kStageBytes;
        const uint32_t vbase = kbase + C::kTileBytes;
        // S = q K^T over 64 keys: sacc[kg][nt] covers keys tok0 + kg*16 + nt*8 ..
        float sacc[4][2][4];
#pragma unroll
        for (int kg = 0; kg < 4; ++kg) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                sacc[kg][nt][0] = sacc[kg][nt][1] = sacc[kg][nt][2] = sacc[kg][nt][3] = 0.f;
            const uint32_t kaddr = kbase + (kg * 16 + k_tok) * C::kPitch + k_col * 2;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(b0, b1, b2, b3, kaddr + kk * 32);
                mma_bf16_16816(sacc[kg][0], qf[kk], b0, b1);
                mma_bf16_16816(sacc[kg][1], qf[kk], b2, b3);
            }
        }
        // scale to the log2 domain; mask keys past each row's position (and
        // past the tile's last key) in tiles that reach the diagonal
        const bool need_mask = tok0 + C::kKeys - 1 > pos_min_block;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int kg = 0; kg < 4; ++kg)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = e >> 1;
                    const int key = tok0 + kg * 16 + nt * 8 + cq + (e & 1);
                    float x = sacc[kg][nt][e] * p.scale_log2;
                    if (need_mask && key > pos[h])
                        x = -INFINITY;
                    sacc[kg][nt][e] = x;
                    mx[h] = fmaxf(mx[h], x);
                }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(kAll, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(kAll, mx[h], 2));
        }
        float base[2], alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float mn = fmaxf(m_run[h], mx[h]);
            base[h] = mn == -INFINITY ? 0.f : mn;
            alpha[h] = exp2f(m_run[h] - base[h]);
            m_run[h] = mn;
        }
        uint32_t pa[4][4];
        float lsum[2] = {0.f, 0.f};
#pragma unroll
        for (int kg = 0; kg < 4; ++kg) {
            pa[kg][0] = pack_bf16x2(exp2f(sacc[kg][0][0] - base[0]), exp2f(sacc[kg][0][1] - base[0]));
            pa[kg][1] = pack_bf16x2(exp2f(sacc[kg][0][2] - base[1]), exp2f(sacc[kg][0][3] - base[1]));
            pa[kg][2] = pack_bf16x2(exp2f(sacc[kg][1][0] - base[0]), exp2f(sacc[kg][1][1] - base[0]));
            pa[kg][3] = pack_bf16x2(exp2f(sacc[kg][1][2] - base[1]), exp2f(sacc[kg][1][3] - base[1]));
            lsum[0] += (bf16_lo(pa[kg][0]) + bf16_hi(pa[kg][0])) +
                       (bf16_lo(pa[kg][2]) + bf16_hi(pa[kg][2]));
            lsum[1] += (bf16_lo(pa[kg][1]) + bf16_hi(pa[kg][1])) +
                       (bf16_lo(pa[kg][3]) + bf16_hi(pa[kg][3]));
        }
        l_run[0] = l_run[0] * alpha[0] + lsum[0];
        l_run[1] = l_run[1] * alpha[1] + lsum[1];
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            oacc[j][0] *= alpha[0];
            oacc[j][1] *= alpha[0];
            oacc[j][2] *= alpha[1];
            oacc[j][3] *= alpha[1];
        }
        // O += P V
#pragma unroll
        for (int kg = 0; kg < 4; ++kg) {
            const uint32_t vaddr = vbase + (kg * 16 + v_tok) * C::kPitch + v_col * 2;
#pragma unroll
            for (int jj = 0; jj < D / 16; ++jj) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(b0, b1, b2, b3, vaddr + jj * 32);
                mma_bf16_16816(oacc[2 * jj], pa[kg], b0, b1);
                mma_bf16_16816(oacc[2 * jj + 1], pa[kg], b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }

    // ---- normalise and store ------------------------------------------------
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(kAll, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(kAll, l_run[h], 2);
    }
    if (aborted)
        return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (pos[h] < 0)
            continue;
        const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
        const int tok = rr[h] / n_rep, hh = rr[h] - tok * n_rep;
        __nv_bfloat16 *o = p.out + ((size_t)(q0 + i0 + tok) * p.Hq + (size_t)g * n_rep + hh) * D + cq;
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            *reinterpret_cast<uint32_t *>(o + 8 * j) =
                pack_bf16x2(oacc[j][2 * h] * inv, oacc[j][2 * h + 1] * inv);
    }
}

template <int D>
cudaError_t launch_prefill_d(const PrefillParams &p, int grid_x, cudaStream_t stream)
{
    using C = PrefillCfg<D>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, p.Hkv);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_kernel<D>, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_prefill(const PrefillParams &p, int D, cudaStream_t stream)
{
    // enough tile slots for any split of total_q tokens over B rows
    const long long slots = ((long long)p.total_q + p.tq - 1) / p.tq + p.B;
    if (slots <= 0)
        return cudaSuccess;
    if (slots > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    if (D == 64)
        return launch_prefill_d<64>(p, (int)slots, stream);
    return launch_prefill_d<128>(p, (int)slots, stream);
}

} // namespace pkv
