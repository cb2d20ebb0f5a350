// pkv_decode.cu -- kernel (2), split-KV paged GQA decode attention, and
// kernel (3), the combine of split partials.
//
// What it computes (AstrAI commit log, page "compare v1.3.12..6f09b1d",
// astrai/extension/attention_ops.py attn_paged_decode and
// attention_backend.py TorchNativeBackend.fwd_decode): for row b, kv head g
// and each of the n_rep = Hq/Hkv query heads h of that group,
//   s_t = scale * <q[b,h], K_t>,  out[b,h] = sum_t softmax(s)_t V_t
// over the row's tokens t, whose K/V rows are found through the page table
// one token at a time (commits by author: "Replace per-tile page lookup
// with per-element lookup in load_tile").  The tokens are cut into splits
// (commits by author: "compute_num_splits", "split partials", "single
// combine kernel"); each split keeps an online max/sum and the splits are
// merged by the combine kernel.
//
// GB300 design of the split kernel (one block per (split, kv head, row)):
//  - each of the NW warps owns an NSTAGE-deep ring of 16-token tiles in
//    shared memory; a tile is 16 K rows + 16 V rows of one kv head, each row
//    a contiguous D*2-byte run in the pool.  Lane t of the warp issues ONE
//    cp.async.bulk (TMA engine) for row t: lanes 0-15 the K rows, 16-31 the
//    V rows, each looked up through the page table on its own, so any
//    page_size works.  Completion is counted on the stage's mbarrier
//    (transaction bytes), so the warp never blocks on a global load.
//  - the warps of a block take the block's tiles round robin and each runs
//    its own online softmax; the block merges the NW warp states in shared
//    memory at the end.
//  - all n_rep query heads of the group are served from the one read of
//    each K/V row: q.K^T and P.V are m16n8k16 bf16 tensor-core products
//    with the (up to 16) query heads as the M rows, fp32 accumulation.
//    Softmax runs in fp32 in the log2 domain; P is rounded to bf16 for the
//    P.V product and the running sum adds those same rounded values.
//  - shared-memory rows are padded by 16 bytes so the ldmatrix reads of 8
//    rows hit 8 distinct 4-bank groups.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr float kLn2 = 0.693147180559945309f;

template <int D>
struct TileShape {
    static constexpr int kTok = 16;                   // tokens per tile
    static constexpr int kRowBytes = D * 2;           // one K or V head row
    static constexpr int kPitch = D * 2 + 16;         // padded smem row
    static constexpr int kStageBytes = 2 * kTok * kPitch;
};

template <int D, int NW, int NSTAGE>
struct SplitCfg {
    using T = TileShape<D>;
    static constexpr int kThreads = NW * 32;
    static constexpr int kRingBytes = NW * NSTAGE * T::kStageBytes;
    // merge area (reuses the ring): NW x 16 rows x D floats + m, l
    static constexpr int kMergeBytes = NW * 16 * D * 4 + 2 * NW * 16 * 4;
    static_assert(kMergeBytes <= kRingBytes, "merge area must fit in the ring");
    static constexpr int kBarOffset = kRingBytes;
    static constexpr int kSmemBytes = kRingBytes + NW * NSTAGE * 8;
};

template <int D, int NW, int NSTAGE>
__global__ void __launch_bounds__(NW * 32)
    split_decode_kernel(const DecodeParams p)
{
    using C = SplitCfg<D, NW, NSTAGE>;
    using T = TileShape<D>;
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int h0 = g * p.n_rep;

    // ---- the row's extent, with the table checked before any use --------
    int L = p.seq_lens[b];
    const int pg0 = p.kv_indptr[b];
    const int pg1 = p.kv_indptr[b + 1];
    unsigned bad = 0;
    if (L < 0 || L > p.max_seq_len) {
        bad |= kFlagBadLen;
        L = L < 0 ? 0 : p.max_seq_len;
    }
    if (pg0 < 0 || pg1 < pg0 || pg1 > p.num_indices) {
        bad |= kFlagBadPage;
        L = 0;
    } else if ((long long)(pg1 - pg0) * p.page_size < (long long)L) {
        bad |= kFlagBadPage;
        L = (pg1 - pg0) * p.page_size;
    }
    if (bad && threadIdx.x == 0 && split == 0 && g == 0)
        atomicOr(p.status, bad);

    const int tok0 = split * p.chunk;
    const int tok1 = min(tok0 + p.chunk, L);
    const int ntok = tok1 - tok0;
    const size_t part_row = (size_t)b * p.Hq + h0;   // first query head of the group

    if (ntok <= 0) {
        if (p.direct) {  // single split and an empty row: zeros
            uint4 *o = reinterpret_cast<uint4 *>(p.out + part_row * D);
            for (int i = threadIdx.x; i < p.n_rep * D / 8; i += blockDim.x)
                o[i] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            for (int r = threadIdx.x; r < p.n_rep; r += blockDim.x) {
                float2 *ml = reinterpret_cast<float2 *>(p.ml_part) +
                             (part_row + r) * p.num_splits + split;
                *ml = make_float2(-INFINITY, 0.f);
            }
        }
        return;
    }

    const int ntiles = (ntok + T::kTok - 1) / T::kTok;
    const int my_tiles = warp < ntiles ? (ntiles - 1 - warp) / NW + 1 : 0;
    unsigned char *ring = smem + warp * NSTAGE * T::kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOffset) + warp * NSTAGE;

    if (lane == 0) {
        for (int st = 0; st < NSTAGE; ++st)
            mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- q fragments: A operand rows = query heads of the group ---------
    const int r = lane >> 2;          // fragment row (and +8)
    const int cq = (lane & 3) * 2;    // fragment column pair
    uint32_t qf[D / 16][4];
    {
        const uint32_t *q0 = reinterpret_cast<const uint32_t *>(p.q + (part_row + r) * D);
        const uint32_t *q1 = reinterpret_cast<const uint32_t *>(p.q + (part_row + r + 8) * D);
        const bool v0 = r < p.n_rep, v1 = r + 8 < p.n_rep;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][0] = v0 ? __ldg(q0 + (kk * 16 + cq) / 2) : 0u;
            qf[kk][1] = v1 ? __ldg(q1 + (kk * 16 + cq) / 2) : 0u;
            qf[kk][2] = v0 ? __ldg(q0 + (kk * 16 + 8 + cq) / 2) : 0u;
            qf[kk][3] = v1 ? __ldg(q1 + (kk * 16 + 8 + cq) / 2) : 0u;
        }
    }

    // ---- producer: lane t copies K row t (t < 16) or V row t-16 ----------
    const int my_t = lane & 15;
    const bool my_v = lane >= 16;
    const __nv_bfloat16 *my_pool = my_v ? p.v_pool : p.k_pool;
    auto issue = [&](int i) {
        const int tile = warp + i * NW;
        const int st = i % NSTAGE;
        const int t0 = tok0 + tile * T::kTok;
        const int nvalid = min(T::kTok, tok1 - t0);
        unsigned char *row = ring + st * T::kStageBytes + (my_v ? T::kTok : 0) * T::kPitch +
                             my_t * T::kPitch;
        if (lane == 0)
            mbar_arrive_expect_tx(&bars[st], (uint32_t)(nvalid * 2 * T::kRowBytes));
        __syncwarp();
        if (my_t < nvalid) {
            const int tok = t0 + my_t;
            int pi, sl;
            if (p.ps_shift >= 0) {
                pi = tok >> p.ps_shift;
                sl = tok & (p.page_size - 1);
            } else {
                pi = tok / p.page_size;
                sl = tok - pi * p.page_size;
            }
            int page = __ldg(p.kv_indices + pg0 + pi);
            if (page < 0 || page >= p.num_pages) {
                atomicOr(p.status, kFlagBadPage);
                page = 0;
            }
            const __nv_bfloat16 *src =
                my_pool + (((size_t)page * p.page_size + sl) * p.Hkv + g) * D;
            bulk_copy_g2s(row, src, T::kRowBytes, &bars[st]);
        } else if (my_v) {
            // V rows past the end must be finite: P is 0 there, 0 * NaN is not.
            uint4 *z = reinterpret_cast<uint4 *>(row);
#pragma unroll
            for (int k = 0; k < T::kRowBytes / 16; ++k)
                z[k] = make_uint4(0u, 0u, 0u, 0u);
        }
    };

    // ---- consumer state ----------------------------------------------------
    float m_run[2] = {-INFINITY, -INFINITY};  // rows r, r+8 (log2 domain)
    float l_run[2] = {0.f, 0.f};              // this lane's share of the sums
    float oacc[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
        oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

    // ldmatrix row addresses (see the fragment layouts of m16n8k16)
    const int k_tok = (lane & 7) + ((lane >> 4) << 3);
    const int k_col = ((lane >> 3) & 1) * 8;
    const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_col = (lane >> 4) * 8;
    const uint32_t ring_s = smem_addr(ring);

    const int npre = min(NSTAGE, my_tiles);
    for (int i = 0; i < npre; ++i)
        issue(i);
    int issued = npre;
    int consumed = 0;
    bool failed = false;

    for (int i = 0; i < my_tiles; ++i) {
        const int st = i % NSTAGE;
        const bool ok = mbar_wait_bounded(&bars[st], (uint32_t)((i / NSTAGE) & 1));
        if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            break;
        }
        consumed = i + 1;
        const int tile = warp + i * NW;
        const int nvalid = min(T::kTok, tok1 - (tok0 + tile * T::kTok));
        const uint32_t kbase = ring_s + st * T::kStageBytes;
        const uint32_t vbase = kbase + T::kTok * T::kPitch;

        // S = Q K^T : 16 heads x 16 tokens, two n8 tiles
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const uint32_t kaddr = kbase + k_tok * T::kPitch + k_col * 2;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(b0, b1, b2, b3, kaddr + kk * 32);
            mma_bf16_16816(sacc[0], qf[kk], b0, b1);
            mma_bf16_16816(sacc[1], qf[kk], b2, b3);
        }

        // online softmax, log2 domain; tokens past the end get -inf
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tt = nt * 8 + cq + (e & 1);
                x[nt][e] = tt < nvalid ? sacc[nt][e] * p.scale_log2 : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m_run[0], mx0);
        const float mn1 = fmaxf(m_run[1], mx1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float alpha0 = exp2f(m_run[0] - base0);
        const float alpha1 = exp2f(m_run[1] - base1);
        m_run[0] = mn0;
        m_run[1] = mn1;

        uint32_t pa[4];
        pa[0] = pack_bf16x2(exp2f(x[0][0] - base0), exp2f(x[0][1] - base0));
        pa[1] = pack_bf16x2(exp2f(x[0][2] - base1), exp2f(x[0][3] - base1));
        pa[2] = pack_bf16x2(exp2f(x[1][0] - base0), exp2f(x[1][1] - base0));
        pa[3] = pack_bf16x2(exp2f(x[1][2] - base1), exp2f(x[1][3] - base1));
        l_run[0] = l_run[0] * alpha0 + ((bf16_lo(pa[0]) + bf16_hi(pa[0])) +
                                        (bf16_lo(pa[2]) + bf16_hi(pa[2])));
        l_run[1] = l_run[1] * alpha1 + ((bf16_lo(pa[1]) + bf16_hi(pa[1])) +
                                        (bf16_lo(pa[3]) + bf16_hi(pa[3])));
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            oacc[j][0] *= alpha0;
            oacc[j][1] *= alpha0;
            oacc[j][2] *= alpha1;
            oacc[j][3] *= alpha1;
        }

        // O += P V : 16 heads x D, one k16 step over the tile's tokens
        const uint32_t vaddr = vbase + v_tok * T::kPitch + v_col * 2;
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(b0, b1, b2, b3, vaddr + jj * 32);
            mma_bf16_16816(oacc[2 * jj], pa, b0, b1);
            mma_bf16_16816(oacc[2 * jj + 1], pa, b2, b3);
        }

        if (i + NSTAGE < my_tiles) {
            __syncwarp();
            fence_proxy_async_smem();
            issue(i + NSTAGE);
            ++issued;
        }
    }

    if (failed) {
        if (lane == 0)
            atomicOr(p.status, kFlagTimeout);
        // let every copy still in flight land before the block can exit
        for (int k = consumed; k < issued; ++k)
            (void)mbar_wait_bounded(&bars[k % NSTAGE], (uint32_t)((k / NSTAGE) & 1));
    }

    // quad-reduce this warp's running sums
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);

    // ---- merge the NW warp states (the ring is free once all warps pass) -
    __syncthreads();
    float *red_o = reinterpret_cast<float *>(smem);   // [NW][16][D]
    float *red_m = red_o + NW * 16 * D;                // [NW][16]
    float *red_l = red_m + NW * 16;                    // [NW][16]
    {
        float *o0 = red_o + (warp * 16 + r) * D + cq;
        float *o1 = o0 + 8 * D;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            *reinterpret_cast<float2 *>(o0 + 8 * j) = make_float2(oacc[j][0], oacc[j][1]);
            *reinterpret_cast<float2 *>(o1 + 8 * j) = make_float2(oacc[j][2], oacc[j][3]);
        }
        if ((lane & 3) == 0) {
            red_m[warp * 16 + r] = failed ? -INFINITY : m_run[0];
            red_m[warp * 16 + r + 8] = failed ? -INFINITY : m_run[1];
            red_l[warp * 16 + r] = failed ? 0.f : l_run[0];
            red_l[warp * 16 + r + 8] = failed ? 0.f : l_run[1];
        }
    }
    __syncthreads();

    const int n_vec = p.n_rep * (D / 4);
    for (int e = threadIdx.x; e < n_vec; e += blockDim.x) {
        const int row = e / (D / 4);
        const int d = (e % (D / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            if (red_l[w * 16 + row] > 0.f)
                M = fmaxf(M, red_m[w * 16 + row]);
        float lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float lw = red_l[w * 16 + row];
            if (!(lw > 0.f))
                continue;
            const float f = exp2f(red_m[w * 16 + row] - M);
            lsum += lw * f;
            const float4 o = *reinterpret_cast<const float4 *>(red_o + (w * 16 + row) * D + d);
            acc.x += o.x * f;
            acc.y += o.y * f;
            acc.z += o.z * f;
            acc.w += o.w * f;
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        if (p.direct) {
            uint2 v;
            v.x = pack_bf16x2(acc.x, acc.y);
            v.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2 *>(p.out + (part_row + row) * D + d) = v;
        } else {
            const size_t slot = (part_row + row) * p.num_splits + split;
            *reinterpret_cast<float4 *>(p.o_part + slot * D + d) = acc;
            if (d == 0)
                reinterpret_cast<float2 *>(p.ml_part)[slot] =
                    lsum > 0.f ? make_float2(M * kLn2, lsum) : make_float2(-INFINITY, 0.f);
        }
    }
}

// ---- combine: one warp per (row, query head) ------------------------------
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p)
{
    constexpr int V = D / 32;   // floats per lane
    const int lane = threadIdx.x & 31;
    const long long bh = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (bh >= (long long)p.B * p.Hq)
        return;
    const int S = p.num_splits;
    const float2 *ml = reinterpret_cast<const float2 *>(p.ml_part) + bh * S;
    const float *o = p.o_part + bh * S * D + lane * V;

    // pass 1: max over non-empty splits, lanes striding over the splits
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) {
        const float2 v = ml[s];
        if (v.y > 0.f)
            M = fmaxf(M, v.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    // pass 2: weights w_s = l_s exp(m_s - M), broadcast 32 at a time
    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = 0.f;
    float den = 0.f;
    constexpr float kLog2e = 1.4426950408889634f;
    for (int s0 = 0; s0 < S; s0 += 32) {
        float w = 0.f;
        if (s0 + lane < S) {
            const float2 v = ml[s0 + lane];
            if (v.y > 0.f)
                w = v.y * exp2f((v.x - M) * kLog2e);
        }
        const int n = min(32, S - s0);
        for (int k = 0; k < n; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            if (wk > 0.f) {
                den += wk;
                const float *src = o + (size_t)(s0 + k) * D;
                if constexpr (V == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(src);
                    acc[0] += wk * x.x;
                    acc[1] += wk * x.y;
                    acc[2] += wk * x.z;
                    acc[3] += wk * x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(src);
                    acc[0] += wk * x.x;
                    acc[1] += wk * x.y;
                }
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16 *dst = p.out + bh * D + lane * V;
    if constexpr (V == 4) {
        uint2 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(dst) = v;
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}

template <int D, int NW, int NSTAGE>
cudaError_t launch_split_cfg(const DecodeParams &p, cudaStream_t stream)
{
    using C = SplitCfg<D, NW, NSTAGE>;
    static DeviceOnce attrs;       // raising the smem limit is per function and device
    const cudaError_t e = attrs.run([] {
        cudaError_t r = cudaFuncSetAttribute(split_decode_kernel<D, NW, NSTAGE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (r != cudaSuccess)
            return r;
        return cudaFuncSetAttribute(split_decode_kernel<D, NW, NSTAGE>,
                                    cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess)
        return e;
    dim3 grid(p.num_splits, p.Hkv, p.B);
    split_decode_kernel<D, NW, NSTAGE><<<grid, C::kThreads, C::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

// Chosen configuration per head dim: 4 warps per block, 3 stages per warp.
constexpr int kNW = 4;
constexpr int kStages = 3;

} // namespace

int split_decode_blocks_per_sm(int D)
{
    const int smem = D == 64 ? SplitCfg<64, kNW, kStages>::kSmemBytes
                             : SplitCfg<128, kNW, kStages>::kSmemBytes;
    const int per_sm = (228 * 1024) / (smem + 1024);   // 1 KB reserved per block
    return per_sm < 1 ? 1 : (per_sm > 8 ? 8 : per_sm);
}

cudaError_t launch_split_decode(const DecodeParams &p, int D, cudaStream_t stream)
{
    if (D == 64)
        return launch_split_cfg<64, kNW, kStages>(p, stream);
    return launch_split_cfg<128, kNW, kStages>(p, stream);
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream)
{
    const long long rows = (long long)p.B * p.Hq;
    const int warps = 8;
    const long long blocks = (rows + warps - 1) / warps;
    if (p.D == 64)
        combine_kernel<64><<<(unsigned)blocks, warps * 32, 0, stream>>>(p);
    else
        combine_kernel<128><<<(unsigned)blocks, warps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace pkv
