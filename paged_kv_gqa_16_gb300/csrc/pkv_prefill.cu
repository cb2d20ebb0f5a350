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
// Layout of the work.  One block of 128 threads takes one (query tile, row,
// kv head): 128 query rows = the tile's 128 / n_rep tokens x the kv head's
// n_rep query heads (token-major).  Thread t owns query row t, which is lane t
// of tensor memory.  Per key tile of 64 tokens:
//  - every thread gathers 16-byte chunks of the tile's K and V rows through
//    the page table with cp.async, straight into the no-swizzle canonical
//    layout the MMA reads (8-row x 16-byte core matrices; consecutive threads
//    fill consecutive 16 bytes), two stages;
//  - one thread issues S = Q K^T (M 128, N 64, K = D in steps of 16; Q and K
//    K-major) into 64 TMEM columns and commits it to an mbarrier;
//  - each thread loads its row of S from TMEM, masks keys past its position,
//    updates its own fp32 online softmax (log2 domain, the scale folded into
//    one FFMA per exponent), writes P (bf16) into shared memory as the K-major
//    A operand, and rescales its row of O in TMEM only when its max has grown
//    by more than 2^8 (P stays below 2^8 otherwise); l sums the fp32 terms;
//  - one thread issues O += P V (M 128, N = D, K = 64; V read MN-major, its
//    rows as they are) into D TMEM columns, then the next tile's S.
// Descriptors: version 1, no swizzle; leading byte offset = stride between
// core matrices along K, stride byte offset = along M/N, for both K-major and
// MN-major operands.  Every mbarrier wait is time-bounded; tensor memory is
// allocated by warp 0 at the start and released on every path.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr unsigned kAllTc = 0xffffffffu;

template <int D>
struct TcCfg {
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
__global__ void __launch_bounds__(TcCfg<D>::kThreads, 2) prefill_tc_kernel(const PrefillParams p)
{
    using C = TcCfg<D>;
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
cudaError_t launch_tc_d(const PrefillParams &p, int max_q_len, cudaStream_t stream)
{
    using C = TcCfg<D>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        attr_done = true;
    }
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D>, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_prefill(const PrefillParams &p, int D, int max_q_len, cudaStream_t stream)
{
    if (D == 64)
        return launch_tc_d<64>(p, max_q_len, stream);
    return launch_tc_d<128>(p, max_q_len, stream);
}

} // namespace pkv
