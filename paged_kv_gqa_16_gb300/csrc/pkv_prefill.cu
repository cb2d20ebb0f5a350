// pkv_prefill.cu -- paged ragged prefill / extend attention on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
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
// A query tile is 128 query rows = 128 / n_rep tokens x the kv head's n_rep
// query heads (token-major) of one (row, kv head); the thread that owns query
// row t of a tile owns lane t of tensor memory.  Per K/V tile of 64 keys:
// K and V rows are gathered through the page table with 16-byte cp.async,
// straight into the no-swizzle canonical layout the MMA reads (8-row x
// 16-byte core matrices); S = Q K^T (M 128, N 64, K = D in steps of 16; Q
// and K K-major) goes to tensor memory; each row's thread reads its row of
// S, masks keys past its position, updates its own fp32 online softmax (log2
// domain, the scale folded into one FFMA per exponent, l from the fp32
// terms), rescales its row of O in tensor memory only when its max has grown
// by more than 2^8, and writes P (bf16) to shared memory as the K-major A
// operand; O += P V (M 128, N = D, K = 64; V read MN-major, its rows as they
// are) accumulates in tensor memory.  Two block layouts, chosen by D:
//
//  - D = 64, prefill_row_kernel: one tile per block of 128 threads, three
//    blocks per SM.  All threads gather (two stages) and run the softmax; one
//    thread issues the MMAs, and the steps alternate within a block while
//    the SM's blocks overlap one another.
//  - D = 128, prefill_pair_kernel: two consecutive tiles (A, B) per block,
//    sharing every K/V tile, with warp roles handing work over through
//    mbarriers: warps 9-12 gather three K/V stages ahead, warp 8 owns tensor
//    memory and issues S_A and S_B of K/V tile kt (two S buffers per tile),
//    then O_A and O_B of tile kt - 1, and warps 0-3 / 4-7 run the softmax of
//    tiles A / B.  While one tile's rows run their softmax, the tensor cores
//    work on the other tile's S and on both tiles' P V.
//
// Descriptors: version 1, no swizzle; leading byte offset = stride between
// core matrices along K, stride byte offset = along M/N, for both K-major and
// MN-major operands.  Every mbarrier wait is time-bounded; tensor memory is
// allocated at the start and released on every path.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr unsigned kAllTc = 0xffffffffu;

template <int D>
struct RowCfg {
    static constexpr int kRows = 128;
    static constexpr int kKeys = 64;
    static constexpr int kThreads = 128;
    static constexpr int kGroup = D * 16;                  // 8 rows x D bf16, canonical
    static constexpr int kQBytes = kRows / 8 * kGroup;
    static constexpr int kKVBytes = kKeys / 8 * kGroup;    // one K or V tile
    static constexpr int kPGroup = kKeys * 16;             // 8 rows x 64 keys
    static constexpr int kPBytes = kRows / 8 * kPGroup;
    static constexpr int kKVOff = kQBytes;                 // stage s: K, then V
    static constexpr int kPOff = kKVOff + 2 * 2 * kKVBytes;
    static constexpr int kBarOff = kPOff + kPBytes;        // mbar S, mbar O
    static constexpr int kTmemSlot = kBarOff + 16;
    static constexpr int kOffOff = kBarOff + 32;           // [2][64] key offsets
    static constexpr int kSmemBytes = kOffOff + 2 * kKeys * 4;
    // two blocks per SM: 2 x (kSmemBytes + 1 KB reserved) <= 228 KB
    static_assert(2 * (kSmemBytes + 1024) <= 233472, "two blocks per SM");
    // S in columns [0, 64), O in [64, 64 + D): 128 columns at D = 64 (so the
    // three blocks that fit an SM's shared memory all get tensor memory), 256
    // at D = 128
    static constexpr uint32_t kTmemCols = D <= 64 ? 128 : 256;
    static constexpr uint32_t kSCol = 0, kOCol = 64;
};

__device__ __forceinline__ void tc_flag(uint32_t *status, unsigned bits)
{
    if (status != nullptr)
        atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// kind::f16 instruction descriptor: f32 accumulate, bf16 A and B.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                     uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
                 "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane: one load and one
// wait in a single asm statement, so no use of the registers can be
// scheduled before the wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64])
{
    uint32_t r[64];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
                   "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
                   "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                   "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
                   "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
                   "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                 "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                 "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
                 "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                 "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                 "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16-byte global -> shared copy; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int D>
__global__ void __launch_bounds__(RowCfg<D>::kThreads, 2) prefill_row_kernel(const PrefillParams p)
{
    using C = RowCfg<D>;
    constexpr int CH = D / 8;                      // 16-byte chunks per row
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bar_s = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *bar_o = bar_s + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kTmemSlot);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5;

    const int b = blockIdx.y / p.Hkv, g = blockIdx.y % p.Hkv;
    const int n_rep = p.n_rep, tq = p.tq;

    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
    }
    grid_dependency_wait();
    // the row's chunk, checked (a bad row is flagged once, by its tile 0)
    const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
    const int L = p.seq_lens[b];
    const int q_len = q1 - q0;
    const bool row_ok = q_len >= 0 && q0 >= 0 && q1 <= p.total_q && L >= 0 &&
                        L <= p.max_seq_len && q_len <= L;
    if (!row_ok) {
        if (blockIdx.x == 0 && g == 0 && tid == 0)
            tc_flag(p.status, kFlagBadLen);
        return;
    }
    const int n_tiles = (q_len + tq - 1) / tq;
    if (n_tiles > (int)gridDim.x && blockIdx.x == 0 && g == 0 && tid == 0)
        tc_flag(p.status, kFlagBadLen);                // chunk longer than max_q_len
    if ((int)blockIdx.x >= n_tiles)
        return;
    const int t = n_tiles - 1 - (int)blockIdx.x;       // last tile (most keys) first
    const int i0 = t * tq;
    const int ntok = min(tq, q_len - i0);
    const int pos_first = L - q_len + i0;
    const int kv_end = pos_first + ntok;
    const int n_kt = (kv_end + C::kKeys - 1) / C::kKeys;
    const int pg0 = p.kv_indptr[b];
    const int npg = p.kv_indptr[b + 1] - pg0;
    const bool table_ok = pg0 >= 0 && npg >= 0 && p.kv_indptr[b + 1] <= p.num_indices &&
                          (long long)npg * p.page_size >= (long long)L;
    if (!table_ok && tid == 0)
        tc_flag(p.status, kFlagBadPage);

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // ---- loads -------------------------------------------------------------
    // Q: row m = token * n_rep + head; element e of this thread: the 16-byte
    // chunk at canonical offset 16 e (row (e & 7) + 8 * group, chunk c).
    const int rows_used = tq * n_rep;
    for (int e = tid; e < C::kRows * CH; e += C::kThreads) {
        const int r8 = e & 7, c = (e >> 3) % CH, grp = (e >> 3) / CH;
        const int m = grp * 8 + r8;
        const int tok = m / n_rep, hh = m - tok * n_rep;
        const bool live = m < rows_used && tok < ntok;
        const __nv_bfloat16 *src =
            live ? p.q + ((size_t)(q0 + i0 + tok) * p.Hq + (size_t)g * n_rep + hh) * D + c * 8
                 : p.q;
        cp_async16(sbase + e * 16, src, live ? 16u : 0u);
    }
    // pool offsets (16-byte units) of a tile's 64 keys, looked up once by
    // threads 0..63 a tile ahead of the copies; all-ones for keys past kv_end
    uint32_t *s_off = reinterpret_cast<uint32_t *>(smem + C::kOffOff);
    auto lookup = [&](int kt) {
        if (tid < C::kKeys) {
            const int tok = kt * C::kKeys + tid;
            uint32_t off = 0xFFFFFFFFu;
            if (tok < kv_end) {
                const int pi = p.ps_shift >= 0 ? (tok >> p.ps_shift) : (tok / p.page_size);
                const int sl = tok - pi * p.page_size;
                int page = table_ok ? __ldg(p.kv_indices + pg0 + pi) : 0;
                if (page < 0 || page >= p.num_pages) {
                    tc_flag(p.status, kFlagBadPage);
                    page = 0;
                }
                off = (uint32_t)((((size_t)page * p.page_size + sl) * p.Hkv + g) * (D / 8));
            }
            s_off[(kt & 1) * C::kKeys + tid] = off;
        }
    };
    // this thread's copies of a tile are NI rounds (element e = tid + 128 i);
    // load_kv issues rounds [i0, i1)
    constexpr int NI = C::kKeys * CH / C::kThreads;
    auto load_kv = [&](int kt, int stage, int i0, int i1) {
        const uint32_t kdst = sbase + C::kKVOff + stage * 2 * C::kKVBytes;
        const uint32_t vdst = kdst + C::kKVBytes;
        const uint32_t *offs = s_off + (kt & 1) * C::kKeys;
        for (int i = i0; i < i1; ++i) {
            const int e = tid + i * C::kThreads;
            const int r8 = e & 7, c = (e >> 3) % CH, grp = (e >> 3) / CH;
            const uint32_t o = offs[grp * 8 + r8];
            const bool live = o != 0xFFFFFFFFu;
            const size_t off = live ? ((size_t)o + c) * 8 : 0;
            cp_async16(kdst + e * 16, p.k_pool + off, live ? 16u : 0u);
            cp_async16(vdst + e * 16, p.v_pool + off, live ? 16u : 0u);
        }
    };
    lookup(0);
    if (n_kt > 1)
        lookup(1);
    __syncthreads();
    load_kv(0, 0, 0, NI);
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_s = tmem + C::kSCol, t_o = tmem + C::kOCol;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    constexpr uint32_t kIdescS = instr_desc(128, C::kKeys, 0);
    constexpr uint32_t kIdescO = instr_desc(128, D, 1);
    const uint32_t q_s = sbase, p_s = sbase + C::kPOff;
    auto issue_s = [&](int stage) {
        const uint32_t k_s = sbase + C::kKVOff + stage * 2 * C::kKVBytes;
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
            umma(t_s, smem_desc(q_s + s * 256, 128, C::kGroup),
                 smem_desc(k_s + s * 256, 128, C::kGroup), kIdescS, s > 0);
    };
    auto issue_o = [&](int stage, bool first) {
        const uint32_t v_s = sbase + C::kKVOff + stage * 2 * C::kKVBytes + C::kKVBytes;
#pragma unroll
        for (int s = 0; s < C::kKeys / 16; ++s)
            umma(t_o, smem_desc(p_s + s * 256, 128, C::kPGroup),
                 smem_desc(v_s + s * 2 * C::kGroup, C::kGroup, 128), kIdescO,
                 (first && s == 0) ? 0u : 1u);
    };
    if (tid == 0) {
        issue_s(0);
        umma_commit(bar_s);
    }

    // this thread's query row
    const int m = tid;
    const int tok_m = m / n_rep;
    const int pos = (m < rows_used && tok_m < ntok) ? pos_first + tok_m : -1;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    unsigned char *p_row = smem + C::kPOff + (m >> 3) * C::kPGroup + (m & 7) * 16;

    for (int kt = 0; kt < n_kt && ok; ++kt) {
        const int stage = kt & 1;
        // S of this tile (and the previous tile's P V) are done
        ok = mbar_wait_bounded(bar_s, (uint32_t)(kt & 1));
        if (!__all_sync(kAllTc, ok)) {
            ok = false;
            if ((tid & 31) == 0)
                tc_flag(p.status, kFlagTimeout);
        }
        ok = __syncthreads_and(ok);
        if (!ok)
            break;
        tc_fence_after();
        // the next tile's copies: half now, the rest spread through the P
        // loop below, so load-store issue overlaps the softmax arithmetic
        const bool more = kt + 1 < n_kt;
        if (more)
            load_kv(kt + 1, stage ^ 1, 0, NI / 2);

        // ---- softmax of this row over the tile's 64 keys ----------------
        const int key0 = kt * C::kKeys;
        const bool need_mask = key0 + C::kKeys - 1 > pos_first;
        // raw scores; the scale (> 0) is applied once to the max and folded
        // into each exponent's FFMA
        float sv[C::kKeys];
        static_assert(C::kKeys == 64, "one 64-column load per tile");
        tmem_ld64(t_s + lane_off, sv);
        if (need_mask) {
#pragma unroll
            for (int i = 0; i < C::kKeys; ++i)
                sv[i] = key0 + i > pos ? -INFINITY : sv[i];
        }
        float mraw = -INFINITY;
#pragma unroll
        for (int i = 0; i < C::kKeys; ++i)
            mraw = fmaxf(mraw, sv[i]);
        const float mx = mraw * p.scale_log2;
        // a new base only when the max grows by more than 2^8 (or first)
        const bool rebase = mx > m_run + 8.f;
        float alpha = 1.f;
        if (rebase) {
            alpha = exp2f(m_run - mx);                 // 0 while m_run is -inf
            m_run = mx;
            l_run *= alpha;
        }
        if (__any_sync(kAllTc, rebase && kt > 0)) {
            // rescale this warp's rows of O (the previous P V has completed)
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
                float v[16];
                tmem_ld16(t_o + lane_off + c0, v);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] *= alpha;
                tmem_st16(t_o + lane_off + c0, v);
            }
            tmem_st_wait();
        }
        const float nbase = m_run == -INFINITY ? 0.f : -m_run;
        const float sl2 = p.scale_log2;
        float lsum = 0.f;
        constexpr int kRest = NI - NI / 2;                // rounds left, kRest | 8
        constexpr int kEvery = (C::kKeys / 8) / kRest;
#pragma unroll
        for (int c = 0; c < C::kKeys / 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float e0 = exp2f(fmaf(sv[c * 8 + 2 * j], sl2, nbase));
                const float e1 = exp2f(fmaf(sv[c * 8 + 2 * j + 1], sl2, nbase));
                w[j] = pack_bf16x2(e0, e1);
                lsum += e0 + e1;                      // l from the fp32 terms
            }
            *reinterpret_cast<uint4 *>(p_row + c * 128) = make_uint4(w[0], w[1], w[2], w[3]);
            if (more && (c + 1) % kEvery == 0) {
                const int i = NI / 2 + (c + 1) / kEvery - 1;
                load_kv(kt + 1, stage ^ 1, i, i + 1);
            }
        }
        cp_async_commit();
        l_run += lsum;

        // ---- hand P (and the next tile) to the tensor cores --------------
        if (kt + 2 < n_kt)
            lookup(kt + 2);                    // published by the barrier below
        cp_async_wait_all();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            issue_o(stage, kt == 0);
            if (kt + 1 < n_kt) {
                issue_s(stage ^ 1);
                umma_commit(bar_s);
            } else {
                umma_commit(bar_o);
            }
        }
    }

    // ---- normalise and store this row -------------------------------------
    bool done = ok && mbar_wait_bounded(bar_o, 0u);
    if (ok && !__all_sync(kAllTc, done) && (tid & 31) == 0)
        tc_flag(p.status, kFlagTimeout);
    done = __syncthreads_and(done);
    tc_fence_after();
    if (done) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        __nv_bfloat16 *orow = nullptr;
        if (pos >= 0) {
            const int hh = m - tok_m * n_rep;
            orow = p.out + ((size_t)(q0 + i0 + tok_m) * p.Hq + (size_t)g * n_rep + hh) * D;
        }
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
            tmem_ld16(t_o + lane_off + c0, v);
            if (orow != nullptr) {
                uint4 lo = make_uint4(pack_bf16x2(v[0] * inv, v[1] * inv),
                                      pack_bf16x2(v[2] * inv, v[3] * inv),
                                      pack_bf16x2(v[4] * inv, v[5] * inv),
                                      pack_bf16x2(v[6] * inv, v[7] * inv));
                uint4 hi = make_uint4(pack_bf16x2(v[8] * inv, v[9] * inv),
                                      pack_bf16x2(v[10] * inv, v[11] * inv),
                                      pack_bf16x2(v[12] * inv, v[13] * inv),
                                      pack_bf16x2(v[14] * inv, v[15] * inv));
                *reinterpret_cast<uint4 *>(orow + c0) = lo;
                *reinterpret_cast<uint4 *>(orow + c0 + 8) = hi;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(C::kTmemCols)
                     : "memory");
}

template <int D>
cudaError_t launch_row(const PrefillParams &p, int max_q_len, cudaStream_t stream)
{
    using C = RowCfg<D>;
    static DeviceOnce attrs;
    const cudaError_t attr_err = attrs.run([] {
        return cudaFuncSetAttribute(prefill_row_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    const long long tiles = ((long long)max_q_len + p.tq - 1) / p.tq;
    const long long rows = (long long)p.B * p.Hkv;
    if (tiles <= 0 || rows <= 0)
        return cudaSuccess;
    if (tiles > 0x7fffffffLL || rows > 65535)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)rows);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_row_kernel<D>, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <int D>
struct PairCfg {
    static constexpr int kRows = 128;                      // query rows of one tile
    static constexpr int kKeys = 64;                       // keys of one K/V tile
    static constexpr int kStages = 3;                      // K/V tiles in flight
    static constexpr int kMmaWarp = 8;                     // warp 8: tensor-memory owner, MMA issue
    static constexpr int kLoadThreads = 128;               // warps 9-12: K/V gathers
    static constexpr int kLoadTid0 = (kMmaWarp + 1) * 32;
    static constexpr int kThreads = kLoadTid0 + kLoadThreads;
    static constexpr int kGroup = D * 16;                  // 8 rows x D bf16, canonical
    static constexpr int kQBytes = kRows / 8 * kGroup;     // one query tile
    static constexpr int kKVBytes = kKeys / 8 * kGroup;    // one K or V tile
    static constexpr int kPGroup = kKeys * 16;             // 8 rows x 64 keys
    static constexpr int kPBytes = kRows / 8 * kPGroup;    // one P tile
    static constexpr int kKVOff = 2 * kQBytes;             // stage s: K, then V
    static constexpr int kPOff = kKVOff + kStages * 2 * kKVBytes;
    static constexpr int kBarOff = kPOff + 2 * kPBytes;
    // mbarriers: kv_full[3], kv_empty[3], s_full[tile][buffer], p_full[2],
    // o_done[2], drain
    static constexpr int kNumBars = 2 * kStages + 9;
    static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
    static constexpr int kAbortOff = kTmemSlot + 4;
    static constexpr int kSmemBytes = kAbortOff + 12;
    static_assert(kSmemBytes <= 232448, "shared memory per block");
    // tensor memory: S of tile X in two buffers at 128 X + 64 j, O of tile X
    // at 256 + D X
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kOCol = 256;
};

// cp.async completion of this thread's earlier copies arrives on bar (the
// barrier's count includes one arrival per loading thread).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

template <int D>
__global__ void __launch_bounds__(PairCfg<D>::kThreads, 1)
    prefill_pair_kernel(const PrefillParams p)
{
    using C = PairCfg<D>;
    constexpr int CH = D / 8;                      // 16-byte chunks per row
    constexpr int NS = C::kStages;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *kv_full = bars, *kv_empty = bars + NS;
    // s_full has one barrier per S buffer, so it never runs two phases ahead
    // of the softmax that waits on it
    uint64_t *s_full = bars + 2 * NS, *p_full = s_full + 4, *o_done = p_full + 2;
    uint64_t *drain = o_done + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kAbortOff);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int b = blockIdx.y / p.Hkv, g = blockIdx.y % p.Hkv;
    const int n_rep = p.n_rep, tq = p.tq;

    grid_dependency_wait();
    // the row's chunk, checked (a bad row is flagged once, by its block 0)
    const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
    const int L = p.seq_lens[b];
    const int q_len = q1 - q0;
    const bool row_ok = q_len >= 0 && q0 >= 0 && q1 <= p.total_q && L >= 0 &&
                        L <= p.max_seq_len && q_len <= L;
    if (!row_ok) {
        if (blockIdx.x == 0 && g == 0 && tid == 0)
            tc_flag(p.status, kFlagBadLen);
        return;
    }
    const int n_tiles = (q_len + tq - 1) / tq;
    if ((n_tiles + 1) / 2 > (int)gridDim.x && blockIdx.x == 0 && g == 0 && tid == 0)
        tc_flag(p.status, kFlagBadLen);                // chunk longer than max_q_len
    // tiles B = n_tiles - 1 - 2x (the most keys first) and A = B - 1
    const int tB = n_tiles - 1 - 2 * (int)blockIdx.x;
    if (tB < 0)
        return;
    const int tA = tB - 1;                             // -1: tile A is idle
    const int kv_end = L - q_len + min(q_len, (tB + 1) * tq);
    const int n_kt = (kv_end + C::kKeys - 1) / C::kKeys;
    const int pg0 = p.kv_indptr[b];
    const int npg = p.kv_indptr[b + 1] - pg0;
    const bool table_ok = pg0 >= 0 && npg >= 0 && p.kv_indptr[b + 1] <= p.num_indices &&
                          (long long)npg * p.page_size >= (long long)L;
    if (!table_ok && tid == 0)
        tc_flag(p.status, kFlagBadPage);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&kv_full[s], C::kLoadThreads);
            mbar_init(&kv_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[2 * x], 1);
            mbar_init(&s_full[2 * x + 1], 1);
            mbar_init(&p_full[x], C::kRows);
            mbar_init(&o_done[x], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Q of both tiles: row m of tile x = token m / n_rep, head m % n_rep
    const int rows_used = tq * n_rep;
    for (int e = tid; e < 2 * C::kRows * CH; e += C::kThreads) {
        const int x = e / (C::kRows * CH), ee = e % (C::kRows * CH);
        const int r8 = ee & 7, c = (ee >> 3) % CH, grp = (ee >> 3) / CH;
        const int m = grp * 8 + r8;
        const int t = x == 0 ? tA : tB;
        const int tok = m / n_rep, hh = m - tok * n_rep;
        const bool live = t >= 0 && m < rows_used && tok < q_len - t * tq;
        const __nv_bfloat16 *src =
            live ? p.q + ((size_t)(q0 + t * tq + tok) * p.Hq + (size_t)g * n_rep + hh) * D + c * 8
                 : p.q;
        cp_async16(sbase + e * 16, src, live ? 16u : 0u);
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (tid >= C::kLoadTid0) {
        // ====================== K/V gathers =================================
        // thread: key lt / 2 of the tile, chunks [CH/2 (lt & 1), CH/2 (lt & 1) + CH/2)
        const int lt = tid - C::kLoadTid0;
        const int key = lt >> 1, c0 = (lt & 1) * (CH / 2);
        const uint32_t row_off = (uint32_t)((key >> 3) * C::kGroup + (key & 7) * 16);
        for (int kt = 0; kt < n_kt; ++kt) {
            const int st = kt % NS;
            if (kt >= NS) {
                const bool ok = mbar_wait_bounded(&kv_empty[st], (uint32_t)(((kt / NS) - 1) & 1));
                if (!ok) {
                    *abort_flag = 1;
                    tc_flag(p.status, kFlagTimeout);
                }
                if (*abort_flag)
                    break;
            }
            const int tok = kt * C::kKeys + key;
            bool live = tok < kv_end;
            size_t off = 0;
            if (live) {
                const int pi = p.ps_shift >= 0 ? (tok >> p.ps_shift) : (tok / p.page_size);
                const int sl = tok - pi * p.page_size;
                int page = table_ok ? __ldg(p.kv_indices + pg0 + pi) : 0;
                if (page < 0 || page >= p.num_pages) {
                    tc_flag(p.status, kFlagBadPage);
                    page = 0;
                }
                off = (((size_t)page * p.page_size + sl) * p.Hkv + g) * D;
            }
            const uint32_t kdst = sbase + C::kKVOff + st * 2 * C::kKVBytes + row_off;
            const uint32_t vdst = kdst + C::kKVBytes;
#pragma unroll
            for (int c = c0; c < c0 + CH / 2; ++c) {
                cp_async16(kdst + c * 128, p.k_pool + off + c * 8, live ? 16u : 0u);
                cp_async16(vdst + c * 128, p.v_pool + off + c * 8, live ? 16u : 0u);
            }
            cp_async_arrive(&kv_full[st]);
        }
        cp_async_wait_all();
    } else if (warp == C::kMmaWarp) {
        // ====================== tensor-core issue ===========================
        constexpr uint32_t kIdescS = instr_desc(128, C::kKeys, 0);
        constexpr uint32_t kIdescO = instr_desc(128, D, 1);
        // Every shared-memory address is below 256 KB, so moving an operand by
        // d bytes adds d / 16 to its descriptor's address field with no carry:
        // the descriptors are built once and offset per stage and k-step.
        const uint64_t dq = smem_desc(sbase, 128, C::kGroup);
        const uint64_t dk = smem_desc(sbase + C::kKVOff, 128, C::kGroup);
        const uint64_t dv = smem_desc(sbase + C::kKVOff + C::kKVBytes, C::kGroup, 128);
        const uint64_t dp = smem_desc(sbase + C::kPOff, 128, C::kPGroup);
        if (lane == 0) {
            auto fail = [&]() {
                *abort_flag = 1;
                tc_flag(p.status, kFlagTimeout);
            };
            bool ok = true;
            for (int kt = 0; kt <= n_kt && ok; ++kt) {
                if (kt < n_kt) {
                    const int st = kt % NS;
                    ok = mbar_wait_bounded(&kv_full[st], (uint32_t)((kt / NS) & 1)) && !*abort_flag;
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint64_t dk_st = dk + (uint64_t)((st * 2 * C::kKVBytes) >> 4);
                    for (int x = 0; x < 2; ++x) {
                        const uint64_t dq_x = dq + (uint64_t)((x * C::kQBytes) >> 4);
                        const uint32_t t_s = tmem + 128 * x + 64 * (kt & 1);
#pragma unroll
                        for (int s = 0; s < D / 16; ++s)
                            umma(t_s, dq_x + 16 * s, dk_st + 16 * s, kIdescS, s > 0);
                        umma_commit(&s_full[2 * x + (kt & 1)]);
                    }
                }
                if (kt > 0) {
                    const int j = kt - 1, sj = j % NS;
                    const uint64_t dv_st = dv + (uint64_t)((sj * 2 * C::kKVBytes) >> 4);
                    for (int x = 0; x < 2 && ok; ++x) {
                        ok = mbar_wait_bounded(&p_full[x], (uint32_t)(j & 1)) && !*abort_flag;
                        if (!ok)
                            break;
                        tc_fence_after();
                        const uint64_t dp_x = dp + (uint64_t)((x * C::kPBytes) >> 4);
                        const uint32_t t_o = tmem + C::kOCol + D * x;
#pragma unroll
                        for (int s = 0; s < C::kKeys / 16; ++s)
                            umma(t_o, dp_x + 16 * s, dv_st + (uint64_t)((s * 2 * C::kGroup) >> 4),
                                 kIdescO, (j == 0 && s == 0) ? 0u : 1u);
                        umma_commit(&o_done[x]);
                    }
                    if (ok)
                        umma_commit(&kv_empty[sj]);
                }
            }
            if (!ok)
                fail();
        }
        __syncwarp();
    } else {
        // ====================== softmax of tile x, row m ====================
        const int x = warp >> 2;
        const int m = tid & (C::kRows - 1);
        const int t = x == 0 ? tA : tB;
        const int tok_m = m / n_rep;
        const int ntok = t >= 0 ? min(tq, q_len - t * tq) : 0;
        const int pos_first = L - q_len + (t >= 0 ? t * tq : 0);
        const int pos = (t >= 0 && m < rows_used && tok_m < ntok) ? pos_first + tok_m : -1;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t t_o = tmem + C::kOCol + D * x;
        unsigned char *p_row =
            smem + C::kPOff + x * C::kPBytes + (m >> 3) * C::kPGroup + (m & 7) * 16;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int kt = 0; kt < n_kt; ++kt) {
            ok = mbar_wait_bounded(&s_full[2 * x + (kt & 1)], (uint32_t)((kt >> 1) & 1)) &&
                 !*abort_flag;
            if (!__all_sync(kAllTc, ok)) {
                ok = false;
                if (lane == 0) {
                    *abort_flag = 1;
                    tc_flag(p.status, kFlagTimeout);
                }
                break;
            }
            tc_fence_after();
            const int key0 = kt * C::kKeys;
            const bool need_mask = key0 + C::kKeys - 1 > pos_first;
            float sv[C::kKeys];
            static_assert(C::kKeys == 64, "one 64-column load per tile");
            tmem_ld64(tmem + 128 * x + 64 * (kt & 1) + lane_off, sv);
            if (need_mask) {
#pragma unroll
                for (int i = 0; i < C::kKeys; ++i)
                    sv[i] = key0 + i > pos ? -INFINITY : sv[i];
            }
            float mraw = -INFINITY;
#pragma unroll
            for (int i = 0; i < C::kKeys; ++i)
                mraw = fmaxf(mraw, sv[i]);
            const float mx = mraw * p.scale_log2;
            // a new base only when the max grows by more than 2^8 (or first)
            const bool rebase = mx > m_run + 8.f;
            float alpha = 1.f;
            if (rebase) {
                alpha = exp2f(m_run - mx);             // 0 while m_run is -inf
                m_run = mx;
                l_run *= alpha;
            }
            // O and P of this tile are free once the previous P V is done
            if (kt > 0) {
                ok = mbar_wait_bounded(&o_done[x], (uint32_t)((kt - 1) & 1)) && !*abort_flag;
                if (!__all_sync(kAllTc, ok)) {
                    ok = false;
                    if (lane == 0) {
                        *abort_flag = 1;
                        tc_flag(p.status, kFlagTimeout);
                    }
                    break;
                }
                tc_fence_after();
            }
            if (__any_sync(kAllTc, rebase && kt > 0)) {
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float v[16];
                    tmem_ld16(t_o + lane_off + c0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        v[i] *= alpha;
                    tmem_st16(t_o + lane_off + c0, v);
                }
                tmem_st_wait();
            }
            const float nbase = m_run == -INFINITY ? 0.f : -m_run;
            const float sl2 = p.scale_log2;
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < C::kKeys / 8; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float e0 = exp2f(fmaf(sv[c * 8 + 2 * jj], sl2, nbase));
                    const float e1 = exp2f(fmaf(sv[c * 8 + 2 * jj + 1], sl2, nbase));
                    w[jj] = pack_bf16x2(e0, e1);
                    lsum += e0 + e1;                  // l from the fp32 terms
                }
                *reinterpret_cast<uint4 *>(p_row + c * 128) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            l_run += lsum;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_full[x]);
        }
        // ---- normalise and store this row ----------------------------------
        if (ok) {
            ok = mbar_wait_bounded(&o_done[x], (uint32_t)((n_kt - 1) & 1)) && !*abort_flag;
            if (!__all_sync(kAllTc, ok) && lane == 0) {
                *abort_flag = 1;
                tc_flag(p.status, kFlagTimeout);
            }
        }
        tc_fence_after();
        if (__all_sync(kAllTc, ok)) {
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            __nv_bfloat16 *orow = nullptr;
            if (pos >= 0) {
                const int hh = m - tok_m * n_rep;
                orow = p.out + ((size_t)(q0 + t * tq + tok_m) * p.Hq + (size_t)g * n_rep + hh) * D;
            }
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
                float v[16];
                tmem_ld16(t_o + lane_off + c0, v);
                if (orow != nullptr) {
                    uint4 lo = make_uint4(pack_bf16x2(v[0] * inv, v[1] * inv),
                                          pack_bf16x2(v[2] * inv, v[3] * inv),
                                          pack_bf16x2(v[4] * inv, v[5] * inv),
                                          pack_bf16x2(v[6] * inv, v[7] * inv));
                    uint4 hi = make_uint4(pack_bf16x2(v[8] * inv, v[9] * inv),
                                          pack_bf16x2(v[10] * inv, v[11] * inv),
                                          pack_bf16x2(v[12] * inv, v[13] * inv),
                                          pack_bf16x2(v[14] * inv, v[15] * inv));
                    *reinterpret_cast<uint4 *>(orow + c0) = lo;
                    *reinterpret_cast<uint4 *>(orow + c0 + 8) = hi;
                }
            }
        }
    }
    // every role is done; on an abort the MMA warp waits (bounded) for the
    // tensor cores to drain before tensor memory is released
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        if (*abort_flag && lane == 0) {
            umma_commit(drain);
            (void)mbar_wait_bounded(drain, 0u);
        }
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(C::kTmemCols)
                     : "memory");
    }
}

template <int D>
cudaError_t launch_pair(const PrefillParams &p, int max_q_len, cudaStream_t stream)
{
    using C = PairCfg<D>;
    static DeviceOnce attrs;
    const cudaError_t attr_err = attrs.run([] {
        return cudaFuncSetAttribute(prefill_pair_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    const long long tiles = ((long long)max_q_len + p.tq - 1) / p.tq;
    const long long pairs = (tiles + 1) / 2;
    const long long rows = (long long)p.B * p.Hkv;
    if (pairs <= 0 || rows <= 0)
        return cudaSuccess;
    if (pairs > 0x7fffffffLL || rows > 65535)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pairs, (unsigned)rows);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_pair_kernel<D>, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_prefill(const PrefillParams &p, int D, int max_q_len, cudaStream_t stream)
{
    // the paired, warp-specialised layout is 27-31% faster at D = 128; at
    // D = 64 the single-tile blocks, three to an SM, are 16% faster
    if (D == 64)
        return launch_row<64>(p, max_q_len, stream);
    return launch_pair<128>(p, max_q_len, stream);
}

} // namespace pkv
