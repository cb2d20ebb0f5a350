// pkv_fused.cu -- the production split-KV decode kernel and its piece
// combine.
//
// What it computes is the same as the split kernel in pkv_decode.cu (AstrAI
// commit log, compare v1.3.12..6f09b1d, attention_ops.py attn_paged_decode):
// out[b, h] = softmax(scale * q[b,h] K^T) V over the row's tokens, K/V of kv
// head h / n_rep gathered token by token through the page table.  How the
// work is cut differs from the pages' grid of (batch, head, split) blocks
// (commits by author, "compute_num_splits ... target 512 blocks"):
//
//  - Persistent and token-balanced.  The grid has G blocks (one per SM).
//    All rows, laid end to end, are cut into G equal contiguous ranges;
//    block c streams range c, which may cover the tail of one row, whole
//    rows and the head of another.  Each (block, row) overlap with tokens is
//    a "piece".  A row weighs its tokens plus a fixed row cost (placed
//    before its first token), so blocks that start more rows stream fewer
//    tokens.  No block waits on another.
//  - All kv heads of a row in one block.  The pool is [page, slot, Hkv, D],
//    so the HPC (<= 8) kv heads handled together are one contiguous run of
//    HPC*D*2 bytes per token (2 KB at Hkv = 8, D = 128).  A producer warp
//    copies one such run per token with cp.async.bulk (TMA engine) into a
//    ring of 16-token stages (K rows, then V rows; rows padded by 16 bytes
//    so ldmatrix reads are bank-conflict free), looked up through the page
//    table token by token.  Full/empty mbarriers hand stages between the
//    producer and the HPC consumer warps; every wait is time-bounded.
//  - One consumer warp per kv head.  It serves that head's n_rep query heads
//    (the M rows of m16n8k16 bf16 tensor-core products) from the shared
//    stage: q.K^T, an fp32 online softmax in the log2 domain, then P.V with
//    P rounded to bf16 and the running sum built from the same rounded P.
//  - A piece that is a whole row writes the bf16 output directly.  Other
//    pieces write (normalised o, m, l) partials to slot (block + row), and
//    the piece combine kernel merges each row's consecutive pieces.
#include <cmath>

#include "pkv_advance.cuh"

namespace pkv {

namespace {

constexpr float kLn2f = 0.693147180559945309f;
constexpr float kLog2ef = 1.4426950408889634f;
// the piece combine splits D until it has about this many items
constexpr long long kCombineMinItems = 128;
constexpr int kSmemLimit = 232448;        // opt-in shared memory per block, sm_100 family
constexpr unsigned kFull = 0xffffffffu;

// Wait for phase `parity` of `bar` (limit_ns as mbar_wait_bounded: zero is one
// non-blocking probe); false if the limit ran out or another warp aborted
// (*abort set).  The abort word is read only once the phase is not already
// complete: a warp that fails stops its part of the pipeline, so every other
// warp's next wait that blocks sees the word.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity,
                                                   unsigned long long limit_ns,
                                                   volatile int *abort)
{
    if (limit_ns == 0)
        return mbar_test_wait(bar, parity) && !*abort;
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort || global_timer_ns() - t0 > limit_ns)
            return false;
    }
    return true;
}

template <int D, int HPC>
struct FusedCfg {
    static constexpr int kTok = 16;
    static constexpr int kThreads = (HPC + 1) * 32;
    static constexpr int kRowBytes = HPC * D * 2;     // one token, HPC kv heads
    static constexpr int kPitch = kRowBytes + 16;
    static constexpr int kStageBytes = 2 * kTok * kPitch;
    static constexpr int kFixedBytes = (kFusedMaxRows + 1) * 4 + 64 + 2 * 8 * 8;
    static constexpr int kStagesFit = (kSmemLimit - kFixedBytes) / kStageBytes;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
    static_assert(kStages >= 2, "ring needs two stages");
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kBarOffset = kRingBytes;                    // full[], empty[]
    static constexpr int kPrefixOffset = kBarOffset + 2 * kStages * 8;
    static constexpr int kScratchOffset = kPrefixOffset + (kFusedMaxRows + 1) * 4;
    // per-row q block and RoPE row, copied ahead by the producer: two
    // mbarriers, the (cos, sin) row, then as many q bytes as fit
    static constexpr int kQBarOffset = (kScratchOffset + 64 + 15) / 16 * 16;
    static constexpr int kCsOffset = kQBarOffset + 16;
    static constexpr int kQOffset = (kCsOffset + D * 4 + 127) / 128 * 128;
    static constexpr int kQWant = 16 * HPC * D * 2;                   // n_rep up to 16
    static constexpr int kQFree = (kSmemLimit - kQOffset) / 128 * 128;
    static constexpr int kQCapBytes = kQWant < kQFree ? kQWant : kQFree;
    static constexpr int kSmemBytes = kQOffset + kQCapBytes;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
    static_assert(kQBarOffset % 16 == 0 && kCsOffset % 16 == 0 && kQOffset % 16 == 0,
                  "bulk-copy destinations and mbarriers need 16-byte alignment");
    static_assert(kBarOffset % 16 == 0 && kPrefixOffset % 16 == 0, "alignment");
};

// Fused step: the stage holds the new token's raw K/V (copied from k_new /
// v_new) in row jn.  This warp rotates its kv head's K slice there (the same
// fp32 arithmetic as the append kernel, so the bits agree), and writes K and
// V to the token's pool slot.  Lane l owns pairs 2l, 2l+1 of the head
// (D = 128) or pair l (D = 64): cs holds their (cos, sin).
template <int D, int kPitch, int kTok>
__device__ __forceinline__ void insert_new_token(const FusedParams &p, unsigned char *stage_col,
                                                 int jn, int lane, int b, int kvh, int tn,
                                                 int page, float4 cs, bool rope_ok)
{
    const bool page_ok = page >= 0 && page < p.num_pages;
    if (lane == 0) {
        if (!page_ok)
            atomicOr(p.status, kFlagBadPage);
        if (!rope_ok)
            atomicOr(p.status, kFlagBadPos);
    }
    unsigned char *krow = stage_col + jn * kPitch;
    unsigned char *vrow = stage_col + (kTok + jn) * kPitch;
    const int pin = p.ps_shift >= 0 ? (tn >> p.ps_shift) : (tn / p.page_size);
    const size_t dst = (((size_t)page * p.page_size + (tn - pin * p.page_size)) * p.Hkv + kvh) * D;
    if constexpr (D == 128) {
        uint2 k = reinterpret_cast<uint2 *>(krow)[lane];
        const uint2 v = reinterpret_cast<const uint2 *>(vrow)[lane];
        if (p.rope != nullptr) {
            if (rope_ok) {
                k.x = rotate_pair(k.x, cs.x, cs.y);
                k.y = rotate_pair(k.y, cs.z, cs.w);
            } else {
                k = make_uint2(0u, 0u);
            }
            reinterpret_cast<uint2 *>(krow)[lane] = k;
        }
        if (page_ok && rope_ok) {
            reinterpret_cast<uint2 *>(p.k_pool_w + dst)[lane] = k;
            reinterpret_cast<uint2 *>(p.v_pool_w + dst)[lane] = v;
        }
    } else {
        uint32_t k = reinterpret_cast<uint32_t *>(krow)[lane];
        const uint32_t v = reinterpret_cast<const uint32_t *>(vrow)[lane];
        if (p.rope != nullptr) {
            k = rope_ok ? rotate_pair(k, cs.x, cs.y) : 0u;
            reinterpret_cast<uint32_t *>(krow)[lane] = k;
        }
        if (page_ok && rope_ok) {
            reinterpret_cast<uint32_t *>(p.k_pool_w + dst)[lane] = k;
            reinterpret_cast<uint32_t *>(p.v_pool_w + dst)[lane] = v;
        }
    }
    // the stage is refilled by bulk copies later: order these generic writes
    // before that async-proxy access, and make them visible to the warp
    fence_proxy_async_smem();
    __syncwarp();
}

// Block owning flattened token x under the partition x in [c*T/G, (c+1)*T/G).
__device__ __forceinline__ int block_of(long long x, long long T, int G)
{
    return (int)(((x + 1) * G + T - 1) / T) - 1;
}

// ---- the partition, shared by the decode kernel and the per-step plan -----
// Token count of virtual row r after the checks: a negative length counts as
// zero, one above max_seq_len as max_seq_len, and a row whose table is
// malformed or does not cover its length is cut to what the table covers.
// The failed checks' flags go to `bad`.
__device__ __forceinline__ int checked_row_len(const FusedParams &p, int r, unsigned &bad)
{
    const int b = r % p.B;
    int L = p.seq_lens[b];
    const int pg0 = p.kv_indptr[b];
    const int pg1 = p.kv_indptr[b + 1];
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
    return L;
}

// prefix[0..Bv] of the rows' partition weights (a non-empty row weighs its
// tokens plus row_cost), computed by every thread of the block; report: OR
// the flags of the first B rows into the status word.
__device__ __forceinline__ void row_prefix(const FusedParams &p, int *prefix, bool report)
{
    const int Bv = p.Bv, lane = threadIdx.x & 31;
    for (int r = threadIdx.x; r < Bv; r += blockDim.x) {
        unsigned bad = 0;
        const int L = checked_row_len(p, r, bad);
        if (bad && report && r < p.B)
            atomicOr(p.status, bad);
        prefix[r + 1] = L > 0 ? L + p.row_cost : 0;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        int carry = 0;
        for (int base = 0; base < Bv; base += 32) {
            const int i = base + lane;
            int v = i < Bv ? prefix[i + 1] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(kFull, v, off);
                if (lane >= off)
                    v += n;
            }
            v += carry;
            if (i < Bv)
                prefix[i + 1] = v;
            carry = __shfl_sync(kFull, v, 31);
        }
        if (lane == 0)
            prefix[0] = 0;
    }
    __syncthreads();
}

// Blocks that get work: at least kFusedMinTokens positions each, at most the
// grid, at least one.
__device__ __forceinline__ unsigned active_blocks(unsigned T, unsigned grid)
{
    unsigned Gu = (T + kFusedMinTokens - 1) / kFusedMinTokens;
    if (Gu > grid)
        Gu = grid;
    return Gu < 1 ? 1 : Gu;
}

// First row whose positions reach past `start` (never an empty row).
__device__ __forceinline__ int first_row(const int *prefix, int Bv, long long start)
{
    int lo = 0, hi = Bv - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)prefix[mid + 1] > start)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// The per-step plan (int32 words): [0] T, [1] active blocks G, [2] grid,
// [3] virtual rows Bv, [4] rows B, [5] page_size, [6..15] unused; then
// prefix[0..Bv] (padded to a multiple of 4 words); then one entry of
// kPlanEntryInts words per block of the grid: [0] its first row r0 (-1: no
// work), [1] the base wb of that row's page-table window, [2] the row's
// first table entry kv_indptr[b], [3] its entry count, [4] and [5] the
// positions of the row's first and last-plus-one token, [6] and [7] the
// block's positions [start, end), [8..71] the window (the row's table
// entries wb .. wb + 63, 0 past the table).
constexpr int kPlanHeaderInts = 16;
constexpr int kPlanEntryInts = 72;

__device__ __forceinline__ const int32_t *plan_entry(const int32_t *plan, int Bv, int c)
{
    return plan + kPlanHeaderInts + ((Bv + 1 + 3) & ~3) + (size_t)c * kPlanEntryInts;
}

template <int D, int HPC>
__global__ void __launch_bounds__(FusedCfg<D, HPC>::kThreads, 1)
    fused_decode_kernel(const FusedParams p)
{
    using C = FusedCfg<D, HPC>;
    constexpr int NST = C::kStages;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);
    uint64_t *empty = full + NST;
    int *prefix = reinterpret_cast<int *>(smem + C::kPrefixOffset);
    volatile int *scratch = reinterpret_cast<volatile int *>(smem + C::kScratchOffset);
    uint64_t *qbar = reinterpret_cast<uint64_t *>(smem + C::kQBarOffset);
    const float *s_cs = reinterpret_cast<const float *>(smem + C::kCsOffset);
    const __nv_bfloat16 *s_q = reinterpret_cast<const __nv_bfloat16 *>(smem + C::kQOffset);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int Bv = p.Bv;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 32);     // every producer lane arrives
            mbar_init(&empty[i], HPC);
        }
        mbar_init(&qbar[0], 1);          // q block landed
        mbar_init(&qbar[1], HPC);        // every consumer has read it
        fence_mbar_init();
        scratch[0] = 0;   // abort flag
    }
    // inputs may come from the kernel just before (the append): wait for it
    grid_dependency_wait();

    // ---- the producer's copy issue, shared by its early start (below) and
    // its row loop.  Lanes 0-15 copy K rows, 16-31 V rows, of one 16-token
    // stage; the page ids come from a 64-entry window of the row's table.
    const int HQVb = HPC * p.n_rep;
    const bool q_staged = HQVb * D * 2 <= C::kQCapBytes;
    auto rope_row_needed = [&](long long lo_, long long hi_) {
        const int pos = (int)(hi_ - lo_) - 1;
        return p.step && p.rope != nullptr && pos < p.rope_max_pos;
    };
    const int my_t = lane & 15;
    const bool my_v = lane >= 16;
    auto page_of_tok = [&](int t) {
        return p.ps_shift >= 0 ? (t >> p.ps_shift) : (t / p.page_size);
    };
    // the row's q block (and RoPE row) into shared memory, by lane 0
    auto stage_q = [&](int b, int hg, long long lo, long long hi) {
        if (lane == 0) {
            const bool need_cs = rope_row_needed(lo, hi);
            const uint32_t qbytes = (uint32_t)(HQVb * D * 2);
            mbar_arrive_expect_tx(&qbar[0], qbytes + (need_cs ? D * 4 : 0));
            bulk_copy_g2s(const_cast<__nv_bfloat16 *>(s_q),
                          p.q + ((size_t)b * p.Hq + (size_t)hg * HQVb) * D, qbytes, &qbar[0]);
            if (need_cs)
                bulk_copy_g2s(const_cast<float *>(s_cs), p.rope + (size_t)(hi - lo - 1) * D,
                              D * 4, &qbar[0]);
        }
    };
    // one stage: tokens tok .. tok + nvalid - 1 of the row piece ending at t1
    // (row length Lrow), into ring stage st
    auto issue_stage = [&](int st, int tok, int t1, int Lrow, int b, size_t head_off, int pg0,
                           int npg, int &wb, int &idx0, int &idx1, uint64_t policy) {
        fence_proxy_async_smem();
        const int nvalid = min(C::kTok, t1 - tok);
        if (page_of_tok(tok) >= wb + 32) {       // slide the window by 32
            wb += 32;
            idx0 = idx1;
            idx1 = wb + 32 + lane < npg ? __ldg(p.kv_indices + pg0 + wb + 32 + lane) : 0;
        }
        unsigned char *row = smem + st * C::kStageBytes +
                             ((my_v ? C::kTok : 0) + my_t) * C::kPitch;
        if (my_v && my_t >= nvalid) {
            // V rows past the piece's end must be finite (P is 0 there)
            uint4 *z = reinterpret_cast<uint4 *>(row);
            for (int k = 0; k < C::kRowBytes / 16; ++k)
                z[k] = make_uint4(0u, 0u, 0u, 0u);
        }
        // every lane joins the shuffles; only lanes with a token use them
        const int t = tok + (my_t < nvalid ? my_t : 0);
        const int pi = page_of_tok(t);
        const int sl = t - pi * p.page_size;
        const int wofs = pi - wb;                  // in [0, 64)
        const int e0 = __shfl_sync(kFull, idx0, wofs & 31);
        const int e1 = __shfl_sync(kFull, idx1, wofs & 31);
        int page = wofs < 32 ? e0 : e1;
        // fused step: the row's last token is this step's new token; its
        // K/V come from k_new / v_new (the consumers rotate K in place)
        const int jn = (p.step && t1 == Lrow && tok + nvalid == t1) ? nvalid - 1 : -1;
        if (lane == 0)
            mbar_arrive_expect_tx(&full[st], (uint32_t)(nvalid * 2 * C::kRowBytes));
        else
            mbar_arrive(&full[st]);
        if (my_t == jn) {
            const __nv_bfloat16 *src =
                (my_v ? p.v_new : p.k_new) + (size_t)b * p.Hkv * D + head_off;
            bulk_copy_g2s(row, src, C::kRowBytes, &full[st]);
        }
        if (my_t < nvalid && my_t != jn) {
            if (page < 0 || page >= p.num_pages) {
                atomicOr(p.status, kFlagBadPage);
                page = 0;
            }
            const __nv_bfloat16 *src = (my_v ? p.v_pool : p.k_pool) +
                                       ((size_t)page * p.page_size + sl) * (size_t)p.Hkv * D +
                                       head_off;
            bulk_copy_g2s_hint(row, src, C::kRowBytes, &full[st], policy);
        }
    };

    // ---- the partition: from the step's plan (one round trip: its prefix
    // sums, and this block's first row, its bounds and page-table window), or
    // computed here from the lengths (the plan's absence, or a plan made for
    // another grid or shape)
    bool planned = false;
    bool early = false;               // producer: the first row's q and first stage issued
    int plan_r0 = 0, plan_wb = 0, plan_w0 = 0, plan_w1 = 0, plan_pg0 = 0, plan_npg = 0;
    if (p.plan != nullptr) {
        const int32_t *pe = plan_entry(p.plan, Bv, cta);
        const int hdr_grid = p.plan[2], hdr_bv = p.plan[3];
        const int hdr_b = p.plan[4], hdr_ps = p.plan[5];
        int e_lo = 0, e_hi = 0, e_start = 0, e_end = 0;
        if (warp == HPC) {
            const int ew = lane < 8 ? pe[lane] : 0;
            plan_w0 = pe[8 + lane];
            plan_w1 = pe[40 + lane];
            plan_r0 = __shfl_sync(kFull, ew, 0);
            plan_wb = __shfl_sync(kFull, ew, 1);
            plan_pg0 = __shfl_sync(kFull, ew, 2);
            plan_npg = __shfl_sync(kFull, ew, 3);
            e_lo = __shfl_sync(kFull, ew, 4);
            e_hi = __shfl_sync(kFull, ew, 5);
            e_start = __shfl_sync(kFull, ew, 6);
            e_end = __shfl_sync(kFull, ew, 7);
        } else {
            for (int i = threadIdx.x; i <= Bv; i += HPC * 32)
                prefix[i] = p.plan[kPlanHeaderInts + i];
            plan_r0 = pe[0];
        }
        planned = hdr_grid == (int)gridDim.x && hdr_bv == Bv && hdr_b == p.B &&
                  hdr_ps == p.page_size;
        if (planned && warp == HPC && plan_r0 >= 0) {
            // Early start: the first row's q block and first stage go out now,
            // from this block's entry alone; the compute warps meanwhile copy
            // the prefix sums and meet this warp at the barrier below.
            const int b = plan_r0 % p.B, hg = plan_r0 / p.B;
            const int t0 = (e_start > e_lo ? e_start : e_lo) - e_lo;
            const int t1 = (e_end < e_hi ? e_end : e_hi) - e_lo;
            if (t1 > t0) {
                // K/V first: the q block is small and lands long before them
                int wb = plan_wb, idx0 = plan_w0, idx1 = plan_w1;
                issue_stage(0, t0, t1, e_hi - e_lo, b, (size_t)hg * HPC * D, plan_pg0,
                            plan_npg, wb, idx0, idx1, policy_evict_first());
                if (q_staged)
                    stage_q(b, hg, e_lo, e_hi);
                early = true;
            }
        }
        __syncthreads();
    }
    if (!planned)
        row_prefix(p, prefix, cta == 0);

    // T: the rows' total weight.  Token t of row r sits at position
    // prefix[r] + row_cost + t; block c owns positions [T c / G, T (c+1) / G).
    // T < 2^31 (the launch bounds rows x (max length + row cost)) and
    // G <= 65536, so 32-bit divisions give these bounds exactly:
    // T c / G = (T / G) c + ((T % G) c) / G.
    const unsigned T = (unsigned)prefix[Bv];
    // fewer blocks when there is little work: at least kFusedMinTokens each
    const unsigned Gu = active_blocks(T, gridDim.x);
    const int G = (int)Gu;

    // rows with no tokens: zero output, no pieces (owner: block r mod grid)
    for (int r = cta; r < Bv; r += gridDim.x) {
        if (prefix[r + 1] == prefix[r]) {
            const int b = r % p.B, hg = r / p.B;
            uint4 *o = reinterpret_cast<uint4 *>(
                p.out + ((size_t)b * p.Hq + (size_t)hg * HPC * p.n_rep) * D);
            for (int i = threadIdx.x; i < HPC * p.n_rep * D / 8; i += blockDim.x)
                o[i] = make_uint4(0u, 0u, 0u, 0u);
            if (threadIdx.x == 0 && !planned) {
                p.row_info[2 * r] = 0;
                p.row_info[2 * r + 1] = 0;
            }
        }
    }
    // An unplanned call leaves its partition behind as the step's plan, for
    // the planned calls of the same step (header and prefix sums: block 0;
    // each block its own entry, the producer below for blocks with work).
    int32_t *plan_e = p.plan_out != nullptr
                          ? const_cast<int32_t *>(plan_entry(p.plan_out, Bv, cta)) : nullptr;
    if (p.plan_out != nullptr && cta == 0) {
        for (int i = threadIdx.x; i <= Bv; i += blockDim.x)
            p.plan_out[kPlanHeaderInts + i] = prefix[i];
        if (threadIdx.x == 0) {
            p.plan_out[0] = (int)T;
            p.plan_out[1] = G;
            p.plan_out[2] = (int)gridDim.x;
            p.plan_out[3] = Bv;
            p.plan_out[4] = p.B;
            p.plan_out[5] = p.page_size;
        }
    }
    if (cta >= G) {
        if (plan_e != nullptr && threadIdx.x == 0)
            plan_e[0] = -1;
        return;
    }
    const unsigned t_q = T / Gu, t_r = T % Gu;
    const long long start = (long long)t_q * cta + t_r * (unsigned)cta / Gu;
    const long long end = (long long)t_q * (cta + 1) + t_r * (unsigned)(cta + 1) / Gu;
    if (start >= end) {
        if (plan_e != nullptr && threadIdx.x == 0)
            plan_e[0] = -1;
        return;
    }

    // first row whose positions reach past start (never an empty row)
    const int r0 = planned ? plan_r0 : first_row(prefix, Bv, start);

    if (warp == HPC) {
        // ======================= producer warp ============================
        // K/V are read once per call: first out of L2, so the page table,
        // q and the partials stay
        const uint64_t stream_policy = policy_evict_first();
        int it = early ? 1 : 0, pc = early && q_staged ? 1 : 0;
        bool aborted = false;
        // the next row's first page-table window, loaded one row ahead
        int n_r = -1, n_idx0 = 0, n_idx1 = 0;
        auto prefetch_window = [&](int from) {
            n_r = -1;
            for (int rr = from; rr < Bv; ++rr) {
                if ((long long)prefix[rr] + p.row_cost >= end)
                    break;
                if (prefix[rr + 1] == prefix[rr])
                    continue;
                const int bb = rr % p.B;
                const int q0 = p.kv_indptr[bb];
                int nq = p.kv_indptr[bb + 1] - q0;
                if (q0 < 0 || nq < 0 || q0 > p.num_indices - nq)
                    nq = 0;                    // a table changed since the plan
                n_idx0 = lane < nq ? __ldg(p.kv_indices + q0 + lane) : 0;
                n_idx1 = 32 + lane < nq ? __ldg(p.kv_indices + q0 + 32 + lane) : 0;
                n_r = rr;
                break;
            }
        };
        for (int r = r0; r < Bv && !aborted; ++r) {
            // [lo, hi): the positions of the row's tokens
            const long long lo = (long long)prefix[r] + p.row_cost, hi = prefix[r + 1];
            if (lo >= end)
                break;
            if (hi == prefix[r])
                continue;
            const bool first_early = early && r == r0;
            const int t0 = (int)((start > lo ? start : lo) - lo);
            const int t1 = (int)((end < hi ? end : hi) - lo);
            const int b = r % p.B, hg = r / p.B;
            int pg0, npg;                                  // npg >= pages the row's tokens use
            if (planned && r == r0) {
                pg0 = plan_pg0;                            // checked by the plan
                npg = plan_npg;
            } else {
                pg0 = p.kv_indptr[b];
                npg = p.kv_indptr[b + 1] - pg0;
                if (pg0 < 0 || npg < 0 || pg0 > p.num_indices - npg)
                    npg = 0;                               // a table changed since the plan
            }
            const size_t head_off = (size_t)hg * HPC * D;
            // page-table window: lane l holds entries wb + l and wb + 32 + l of
            // the row, loaded one window ahead of use; a 16-token tile spans at
            // most 17 consecutive entries, which always lie inside the window
            int wb = (page_of_tok(t0) >> 5) << 5;
            int idx0, idx1;
            if (planned && r == r0 && wb == plan_wb) {
                idx0 = plan_w0;
                idx1 = plan_w1;
            } else if (n_r == r && wb == 0) {
                idx0 = n_idx0;
                idx1 = n_idx1;
            } else {
                idx0 = wb + lane < npg ? __ldg(p.kv_indices + pg0 + wb + lane) : 0;
                idx1 = wb + 32 + lane < npg ? __ldg(p.kv_indices + pg0 + wb + 32 + lane) : 0;
            }
            if (plan_e != nullptr && r == r0) {
                // this block's plan entry: its first row, that row's bounds and
                // the page-table window its first stage reads
                plan_e[8 + lane] = idx0;
                plan_e[40 + lane] = idx1;
                if (lane < 8) {
                    const long long v = lane == 0 ? r0 : lane == 1 ? wb : lane == 2 ? pg0
                                      : lane == 3 ? npg : lane == 4 ? lo : lane == 5 ? hi
                                      : lane == 6 ? start : end;
                    plan_e[lane] = (int)v;
                }
            }
            // stage the row's q block (and RoPE row) for the consumers
            if (q_staged && !first_early) {
                if (pc > 0) {
                    const bool ok = mbar_wait_or_abort(&qbar[1], (uint32_t)((pc - 1) & 1), p.handoff_wait_ns, scratch);
                    if (!__all_sync(kFull, ok)) {
                        aborted = true;
                        if (lane == 0) {
                            scratch[0] = 1;
                            atomicOr(p.status, kFlagTimeout);
                        }
                        break;
                    }
                }
                stage_q(b, hg, lo, hi);
                ++pc;
            }
            prefetch_window(r + 1);
            // (the early start issued the first row's first stage already)
            for (int tok = t0 + (first_early ? C::kTok : 0); tok < t1; tok += C::kTok, ++it) {
                const int st = it % NST;
                if (it >= NST) {
                    const bool ok = mbar_wait_or_abort(&empty[st], (uint32_t)(((it / NST) - 1) & 1), p.handoff_wait_ns, scratch);
                    if (!__all_sync(kFull, ok)) {
                        aborted = true;
                        if (lane == 0) {
                            scratch[0] = 1;
                            atomicOr(p.status, kFlagTimeout);
                        }
                        break;
                    }
                }
                issue_stage(st, tok, t1, (int)(hi - lo), b, head_off, pg0, npg, wb, idx0, idx1,
                            stream_policy);
            }
        }
        // Let the copies already issued land before this warp exits, with the
        // full time limit.  Always, not only when this warp gave up: a
        // consumer that gave up waiting skips its stages, and the block must
        // not exit while a copy into its shared memory is in flight.  In a
        // run without timeouts these phases have completed or are about to.
        for (int k = (it > NST ? it - NST : 0); k < it; ++k)
            (void)mbar_wait_bounded(&full[k % NST], (uint32_t)((k / NST) & 1));
        if (pc > 0)
            (void)mbar_wait_bounded(&qbar[0], (uint32_t)((pc - 1) & 1));
        // the piece combine may be scheduled once every block has signalled;
        // signalling at the end (not the start) keeps its blocks from piling
        // onto the first SMs to free up
        grid_launch_dependents();
        return;
    }

    // ========================= consumer warps ===============================
    const int HQV = HPC * p.n_rep;          // query heads per virtual row
    const int fr = lane >> 2;               // fragment row (and fr + 8)
    const int cq = (lane & 3) * 2;          // fragment column pair
    const int k_tok = (lane & 7) + ((lane >> 4) << 3);
    const int k_col = ((lane >> 3) & 1) * 8;
    const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_col = (lane >> 4) * 8;
    const uint32_t smem_s = smem_addr(smem);
    const uint32_t col_off = (uint32_t)(warp * D * 2);
    int it = 0, pc = 0;
    bool aborted = false;

    for (int r = r0; r < Bv; ++r) {
        const long long lo = (long long)prefix[r] + p.row_cost, hi = prefix[r + 1];
        if (lo >= end)
            break;
        if (hi == prefix[r])
            continue;
        const int t0 = (int)((start > lo ? start : lo) - lo);
        const int t1 = (int)((end < hi ? end : hi) - lo);
        const int b = r % p.B, hg = r / p.B;
        const int kvh = hg * HPC + warp;
        const size_t qrow0 = (size_t)b * p.Hq + (size_t)kvh * p.n_rep;
        const int first = block_of(lo, T, G);
        const int last = block_of(hi - 1, T, G);
        if (t0 == 0 && warp == 0 && lane == 0 && !planned) {
            p.row_info[2 * r] = first;
            p.row_info[2 * r + 1] = last - first + 1;
        }

        uint32_t qf[D / 16][4];
        {
            const bool v0 = fr < p.n_rep, v1 = fr + 8 < p.n_rep;
            const bool rot = rope_row_needed(lo, hi);
            const int pos = (int)(hi - lo) - 1;
            const uint32_t *q0, *q1;
            const float2 *cs;
            if (q_staged) {
                // staged by the producer when it started this row
                if (!aborted) {
                    const bool ok = mbar_wait_or_abort(&qbar[0], (uint32_t)(pc & 1), p.handoff_wait_ns, scratch);
                    if (!__all_sync(kFull, ok)) {
                        aborted = true;
                        if (lane == 0) {
                            scratch[0] = 1;
                            atomicOr(p.status, kFlagTimeout);
                        }
                    }
                }
                const size_t lrow = (size_t)warp * p.n_rep + fr;
                q0 = reinterpret_cast<const uint32_t *>(s_q + lrow * D);
                q1 = reinterpret_cast<const uint32_t *>(s_q + (lrow + 8) * D);
                cs = reinterpret_cast<const float2 *>(s_cs);
            } else {
                q0 = reinterpret_cast<const uint32_t *>(p.q + (qrow0 + fr) * D);
                q1 = reinterpret_cast<const uint32_t *>(p.q + (qrow0 + fr + 8) * D);
                cs = reinterpret_cast<const float2 *>(p.rope + (size_t)(rot ? pos : 0) * D);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                qf[kk][0] = v0 ? q0[(kk * 16 + cq) / 2] : 0u;
                qf[kk][1] = v1 ? q1[(kk * 16 + cq) / 2] : 0u;
                qf[kk][2] = v0 ? q0[(kk * 16 + 8 + cq) / 2] : 0u;
                qf[kk][3] = v1 ? q1[(kk * 16 + 8 + cq) / 2] : 0u;
            }
            // fused step: rotate q by the new token's position.  Each 32-bit
            // word is one interleaved pair; words 0/1 hold pair kk*8 + lane%4,
            // words 2/3 pair kk*8 + 4 + lane%4 (rows fr and fr + 8).
            if (rot) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const float2 ca = cs[kk * 8 + (lane & 3)];
                    const float2 cb = cs[kk * 8 + 4 + (lane & 3)];
                    qf[kk][0] = rotate_pair(qf[kk][0], ca.x, ca.y);
                    qf[kk][1] = rotate_pair(qf[kk][1], ca.x, ca.y);
                    qf[kk][2] = rotate_pair(qf[kk][2], cb.x, cb.y);
                    qf[kk][3] = rotate_pair(qf[kk][3], cb.x, cb.y);
                }
            }
            if (q_staged) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&qbar[1]);
                ++pc;
            }
        }
        // fused step, piece ending the row: prefetch what the new token needs
        // (its slot's page and the (cos, sin) of this lane's two pairs)
        const int Lrow = (int)(hi - lo);
        const bool has_new = p.step && t1 == Lrow;
        int new_page = -1;
        float4 new_cs = make_float4(1.f, 0.f, 1.f, 0.f);
        bool new_rope_ok = true;
        if (has_new) {
            const int tn = Lrow - 1;
            const int pin = p.ps_shift >= 0 ? (tn >> p.ps_shift) : (tn / p.page_size);
            const int e0 = p.kv_indptr[b], e1 = p.kv_indptr[b + 1];
            // (a table changed since the plan: no page, flagged at the write)
            new_page = e0 >= 0 && pin < e1 - e0 && e1 <= p.num_indices
                           ? __ldg(p.kv_indices + e0 + pin) : -1;
            if (p.rope != nullptr) {
                new_rope_ok = tn < p.rope_max_pos;
                if (new_rope_ok) {
                    const float *row = p.rope + (size_t)tn * D;
                    if constexpr (D == 128) {
                        new_cs = __ldg(reinterpret_cast<const float4 *>(row) + lane);
                    } else {
                        const float2 c2 = __ldg(reinterpret_cast<const float2 *>(row) + lane);
                        new_cs = make_float4(c2.x, c2.y, 1.f, 0.f);
                    }
                }
            }
        }

        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        float oacc[D / 8][4];
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

        for (int tok = t0; tok < t1; tok += C::kTok, ++it) {
            const int st = it % NST;
            if (!aborted) {
                const bool ok = mbar_wait_or_abort(&full[st], (uint32_t)((it / NST) & 1), p.handoff_wait_ns, scratch);
                if (!__all_sync(kFull, ok)) {
                    aborted = true;
                    if (lane == 0) {
                        scratch[0] = 1;
                        atomicOr(p.status, kFlagTimeout);
                    }
                }
            }
            if (!aborted) {
                const int nvalid = min(C::kTok, t1 - tok);
                const uint32_t kbase = smem_s + st * C::kStageBytes + col_off;
                const uint32_t vbase = kbase + C::kTok * C::kPitch;
                if (has_new && tok + nvalid == t1)
                    insert_new_token<D, C::kPitch, C::kTok>(
                        p, smem + st * C::kStageBytes + warp * D * 2, nvalid - 1, lane, b,
                        kvh, Lrow - 1, new_page, new_cs, new_rope_ok);

                float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                const uint32_t kaddr = kbase + k_tok * C::kPitch + k_col * 2;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(b0, b1, b2, b3, kaddr + kk * 32);
                    mma_bf16_16816(sacc[0], qf[kk], b0, b1);
                    mma_bf16_16816(sacc[1], qf[kk], b2, b3);
                }
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
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
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
                const uint32_t vaddr = vbase + v_tok * C::kPitch + v_col * 2;
#pragma unroll
                for (int jj = 0; jj < D / 16; ++jj) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(b0, b1, b2, b3, vaddr + jj * 32);
                    mma_bf16_16816(oacc[2 * jj], pa, b0, b1);
                    mma_bf16_16816(oacc[2 * jj + 1], pa, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[st]);
        }

        // ---- end of the piece ----------------------------------------------
        l_run[0] += __shfl_xor_sync(kFull, l_run[0], 1);
        l_run[0] += __shfl_xor_sync(kFull, l_run[0], 2);
        l_run[1] += __shfl_xor_sync(kFull, l_run[1], 1);
        l_run[1] += __shfl_xor_sync(kFull, l_run[1], 2);
        const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
        const float inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
        const bool w0 = fr < p.n_rep, w1 = fr + 8 < p.n_rep;
        if (first == last) {
            __nv_bfloat16 *o0 = p.out + (qrow0 + fr) * D + cq;
            __nv_bfloat16 *o1 = p.out + (qrow0 + fr + 8) * D + cq;
#pragma unroll
            for (int j = 0; j < D / 8; ++j) {
                if (w0)
                    *reinterpret_cast<uint32_t *>(o0 + 8 * j) =
                        pack_bf16x2(oacc[j][0] * inv0, oacc[j][1] * inv0);
                if (w1)
                    *reinterpret_cast<uint32_t *>(o1 + 8 * j) =
                        pack_bf16x2(oacc[j][2] * inv1, oacc[j][3] * inv1);
            }
        } else {
            const size_t slot0 = (size_t)(cta + r) * HQV + (size_t)warp * p.n_rep + fr;
            float *o0 = p.o_part + slot0 * D + cq;
            float *o1 = o0 + 8 * (size_t)D;
#pragma unroll
            for (int j = 0; j < D / 8; ++j) {
                if (w0)
                    *reinterpret_cast<float2 *>(o0 + 8 * j) =
                        make_float2(oacc[j][0] * inv0, oacc[j][1] * inv0);
                if (w1)
                    *reinterpret_cast<float2 *>(o1 + 8 * j) =
                        make_float2(oacc[j][2] * inv1, oacc[j][3] * inv1);
            }
            if ((lane & 3) == 0) {
                float2 *ml = reinterpret_cast<float2 *>(p.ml_part);
                if (w0)
                    ml[slot0] = l_run[0] > 0.f ? make_float2(m_run[0] * kLn2f, l_run[0])
                                               : make_float2(-INFINITY, 0.f);
                if (w1)
                    ml[slot0 + 8] = l_run[1] > 0.f ? make_float2(m_run[1] * kLn2f, l_run[1])
                                                   : make_float2(-INFINITY, 0.f);
            }
        }
    }
    grid_launch_dependents();
}

// ---- the per-step plan ------------------------------------------------------
// The partition the decode kernel would compute at its start, written once
// for every call of a step (commits by author, the decode metadata built
// once per step and reused by every layer): the prefix sums, each row's
// first block and piece count (row_info, read by the piece combine), and for
// every block its first row and that row's page-table window.  A planned
// decode call then starts its copies after one round trip to memory instead
// of three.  One block per decode block; dynamic shared memory: Bv + 1 ints.
__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const FusedParams p,
                                                                   int32_t *plan)
{
    extern __shared__ int pl_prefix[];
    const int Bv = p.Bv, cta = blockIdx.x, tid = threadIdx.x;
    grid_dependency_wait();
    row_prefix(p, pl_prefix, cta == 0);
    const unsigned T = (unsigned)pl_prefix[Bv];
    const unsigned Gu = active_blocks(T, gridDim.x);
    const int G = (int)Gu;
    if (cta == 0) {
        for (int i = tid; i <= Bv; i += blockDim.x)
            plan[kPlanHeaderInts + i] = pl_prefix[i];
        for (int r = tid; r < Bv; r += blockDim.x) {
            const long long lo = (long long)pl_prefix[r] + p.row_cost, hi = pl_prefix[r + 1];
            int first = 0, n = 0;
            if (hi != pl_prefix[r]) {
                first = block_of(lo, T, G);
                n = block_of(hi - 1, T, G) - first + 1;
            }
            p.row_info[2 * r] = first;
            p.row_info[2 * r + 1] = n;
        }
        if (tid == 0) {
            plan[0] = (int)T;
            plan[1] = G;
            plan[2] = (int)gridDim.x;
            plan[3] = Bv;
            plan[4] = p.B;
            plan[5] = p.page_size;
        }
    }
    int32_t *e = const_cast<int32_t *>(plan_entry(plan, Bv, cta));
    const unsigned t_q = T / Gu, t_r = T % Gu;
    const long long start = (long long)t_q * cta + t_r * (unsigned)cta / Gu;
    const long long end = (long long)t_q * (cta + 1) + t_r * (unsigned)(cta + 1) / Gu;
    if (cta >= G || start >= end) {
        if (tid == 0)
            e[0] = -1;
        return;
    }
    const int r0 = first_row(pl_prefix, Bv, start);
    const long long lo = (long long)pl_prefix[r0] + p.row_cost;
    const int t0 = (int)((start > lo ? start : lo) - lo);
    const int b = r0 % p.B;
    const int pg0 = p.kv_indptr[b];
    const int npg = p.kv_indptr[b + 1] - pg0;        // checked by row_prefix
    const int pi = p.ps_shift >= 0 ? (t0 >> p.ps_shift) : (t0 / p.page_size);
    const int wb = (pi >> 5) << 5;
    if (tid < 64)
        e[8 + tid] = wb + tid < npg ? __ldg(p.kv_indices + pg0 + wb + tid) : 0;
    if (tid == 0) {
        e[0] = r0;
        e[1] = wb;
        e[2] = pg0;
        e[3] = npg;
        e[4] = (int)lo;
        e[5] = pl_prefix[r0 + 1];
        e[6] = (int)start;
        e[7] = (int)end;
    }
}

// ---- merge the pieces of every row that has more than one ------------------
// An item is one (virtual row, query head, column slice of D / DS): a group
// of WPH warps merges it.  Warp w takes pieces w, w + WPH, ... in rounds of
// U, loaded together; each round rescales the running (M, den, acc) once to
// the round's max and adds the round's weights, which are independent of one
// another.  The group then merges its warps' states in shared memory.  A
// column split (DS > 1) spreads rows with many pieces over more blocks.
template <int D, int WPH, int DS>
__global__ void __launch_bounds__(WPH > 8 ? 32 * WPH : 256)
    piece_combine_kernel(const PieceCombineParams p)
{
    constexpr int DW = D / DS;                         // columns of one item
    constexpr int V = DW / 32;                         // floats per lane
    static_assert(V == 1 || V == 2 || V == 4, "slice width");
    constexpr int U = WPH >= 16 ? 16 : 8;              // pieces loaded ahead per warp
    constexpr int NWARP = WPH > 8 ? WPH : 8;
    constexpr int GROUPS = NWARP / WPH;                // items per block
    __shared__ float s_m[NWARP], s_den[NWARP];
    __shared__ __align__(16) float s_acc[NWARP][DW];
    // the next kernel (the next step's decode) may be scheduled once every
    // block of this grid has started; it waits for this grid's completion
    // before it reads anything this grid writes
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int grp = warp / WPH, wi = warp % WPH;
    const long long item = (long long)blockIdx.x * GROUPS + grp;
    const bool live = item < (long long)p.Bv * p.HQV * DS && !(p.adv.seq_lens != nullptr &&
                                                               blockIdx.x == gridDim.x - 1);
    int n = 0, first = 0, r = 0, j = 0, col = lane * V;
    if (live) {
        const long long pair = item / DS;
        r = (int)(pair / p.HQV);
        j = (int)(pair % p.HQV);
        col += (int)(item % DS) * DW;
    }
    // With a plan, each row's first block and piece count were written by the
    // plan kernel, which completed before the decode grid passed its own
    // wait: read them while the decode grid finishes.  Without one the decode
    // grid writes them: read them after the wait.
    if (p.planned && live) {
        first = p.row_info[2 * r];
        n = p.row_info[2 * r + 1];
    }
    grid_dependency_wait();
    // paged_decode_step_advance: the last block advances the metadata for the
    // next step; the decode grid, the only reader of it, has completed
    if (p.adv.seq_lens != nullptr && blockIdx.x == gridDim.x - 1) {
        advance_block(p.adv);
        return;
    }
    if (!p.planned && live) {
        first = p.row_info[2 * r];
        n = p.row_info[2 * r + 1];
    }
    const float2 *ml = reinterpret_cast<const float2 *>(p.ml_part);
    float M = -INFINITY, den = 0.f;
    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = 0.f;
    if (n > 1) {
        for (int k0 = wi; k0 < n; k0 += WPH * U) {
            float2 mlv[U];
            float o[U][V];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u * WPH;
                if (k < n) {
                    const size_t slot = (size_t)(first + k + r) * p.HQV + j;
                    mlv[u] = __ldcg(ml + slot);
                    const float *src = p.o_part + slot * D + col;
                    if constexpr (V == 4) {
                        const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
                        o[u][0] = x.x; o[u][1] = x.y; o[u][2] = x.z; o[u][3] = x.w;
                    } else if constexpr (V == 2) {
                        const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
                        o[u][0] = x.x; o[u][1] = x.y;
                    } else {
                        o[u][0] = __ldcg(src);
                    }
                } else {
                    mlv[u] = make_float2(-INFINITY, 0.f);
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        o[u][v] = 0.f;
                }
            }
            // the round's max over its pieces with a nonzero sum (an empty
            // piece leaves its o slot unwritten)
            float mr = -INFINITY;
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (mlv[u].y > 0.f)
                    mr = fmaxf(mr, mlv[u].x);
            if (mr == -INFINITY)
                continue;
            const float mn = fmaxf(M, mr);
            const float a = M == -INFINITY ? 0.f : exp2f((M - mn) * kLog2ef);
            den *= a;
#pragma unroll
            for (int v = 0; v < V; ++v)
                acc[v] *= a;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!(mlv[u].y > 0.f))
                    continue;
                const float w = mlv[u].y * exp2f((mlv[u].x - mn) * kLog2ef);
                den += w;
#pragma unroll
                for (int v = 0; v < V; ++v)
                    acc[v] = fmaf(w, o[u][v], acc[v]);
            }
            M = mn;
        }
    }
    if constexpr (WPH > 1) {
        if (lane == 0) {
            s_m[warp] = M;
            s_den[warp] = den;
        }
        if constexpr (V == 4)
            *reinterpret_cast<float4 *>(&s_acc[warp][lane * 4]) =
                make_float4(acc[0], acc[1], acc[2], acc[3]);
        else if constexpr (V == 2)
            *reinterpret_cast<float2 *>(&s_acc[warp][lane * 2]) = make_float2(acc[0], acc[1]);
        else
            s_acc[warp][lane] = acc[0];
        __syncthreads();
        if (wi != 0)
            return;
        float Mg = -INFINITY;
#pragma unroll
        for (int w = 0; w < WPH; ++w)
            if (s_den[grp * WPH + w] > 0.f)
                Mg = fmaxf(Mg, s_m[grp * WPH + w]);
        den = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v)
            acc[v] = 0.f;
#pragma unroll
        for (int w = 0; w < WPH; ++w) {
            const int ww = grp * WPH + w;
            if (!(s_den[ww] > 0.f))
                continue;
            const float f = exp2f((s_m[ww] - Mg) * kLog2ef);
            den += s_den[ww] * f;
#pragma unroll
            for (int v = 0; v < V; ++v)
                acc[v] += s_acc[ww][lane * V + v] * f;
        }
    }
    if (n <= 1)
        return;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int b = r % p.B, hg = r / p.B;
    __nv_bfloat16 *dst = p.out + ((size_t)b * p.Hq + (size_t)hg * p.HQV + j) * D + col;
    if constexpr (V == 4) {
        uint2 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(dst) = v;
    } else if constexpr (V == 2) {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    } else {
        *dst = __float2bfloat16_rn(acc[0] * inv);
    }
}

template <typename Kernel, typename... Params>
cudaError_t launch_pdl(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const Params &...p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p...);
}

template <int D, int HPC>
cudaError_t launch_fused_cfg(const FusedParams &p, int grid, cudaStream_t stream)
{
    using C = FusedCfg<D, HPC>;
    static DeviceOnce attrs;
    cudaError_t e = attrs.run([] {
        cudaError_t r = cudaFuncSetAttribute(fused_decode_kernel<D, HPC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (r != cudaSuccess)
            return r;
        return cudaFuncSetAttribute(fused_decode_kernel<D, HPC>,
                                    cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess)
        return e;
    e = launch_pdl(fused_decode_kernel<D, HPC>, dim3(grid), dim3(C::kThreads),
                               C::kSmemBytes, stream, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_fused_d(const FusedParams &p, int grid, cudaStream_t stream)
{
    switch (p.hpc) {
    case 8:
        return launch_fused_cfg<D, 8>(p, grid, stream);
    case 4:
        return launch_fused_cfg<D, 4>(p, grid, stream);
    case 2:
        return launch_fused_cfg<D, 2>(p, grid, stream);
    default:
        return launch_fused_cfg<D, 1>(p, grid, stream);
    }
}

} // namespace

int fused_heads_per_block(int Hkv)
{
    if (Hkv % 8 == 0)
        return 8;
    if (Hkv % 4 == 0)
        return 4;
    if (Hkv % 2 == 0)
        return 2;
    return 1;
}

namespace {
std::atomic<unsigned long long> g_handoff_wait_ns{kWaitLimitNs};
} // namespace

unsigned long long handoff_wait_ns()
{
    return g_handoff_wait_ns.load(std::memory_order_relaxed);
}

cudaError_t launch_fused_decode(const FusedParams &params, int D, int grid,
                                cudaStream_t stream)
{
    FusedParams p = params;
    p.handoff_wait_ns = handoff_wait_ns();
    if (D == 64)
        return launch_fused_d<64>(p, grid, stream);
    return launch_fused_d<128>(p, grid, stream);
}

} // namespace pkv

extern "C" pkv_status pkv_testing_set_handoff_wait_ns(unsigned long long ns)
{
    if (ns > pkv::kWaitLimitNs)
        return PKV_ERR_INVALID_ARG;
    pkv::g_handoff_wait_ns.store(ns, std::memory_order_relaxed);
    return PKV_OK;
}

namespace pkv {

cudaError_t launch_decode_plan(const FusedParams &p, int grid, int32_t *plan,
                               cudaStream_t stream)
{
    const size_t smem = ((size_t)p.Bv + 1) * sizeof(int);
    cudaError_t e = launch_pdl(decode_plan_kernel, dim3(grid), dim3(kPlanThreads), smem, stream,
                               p, plan);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

cudaError_t launch_piece_combine(const PieceCombineParams &p, int D, int grid_blocks,
                                 cudaStream_t stream)
{
    // warps per item: enough that each warp loads all its pieces in one
    // round; rows are uneven, so size for three times the average pieces
    // per row
    const long long expect = 3 * (grid_blocks / (p.Bv > 0 ? p.Bv : 1)) + 2;
    const int wph = expect <= 8 ? 1 : expect <= 16 ? 2 : expect <= 32 ? 4 : expect <= 64 ? 8 : 16;
    const long long pairs = (long long)p.Bv * p.HQV;
    // split the columns while there are fewer items than about one per SM
    // (few rows, many pieces each: long contexts)
    int ds = 1;
    while (ds < D / 32 && pairs * ds < kCombineMinItems)
        ds *= 2;
    const int warps = wph > 8 ? wph : 8;
    const int groups = warps / wph;
    const unsigned blocks = (unsigned)((pairs * ds + groups - 1) / groups) +
                            (p.adv.seq_lens != nullptr ? 1u : 0u);
    cudaError_t e = cudaErrorInvalidValue;
#define PKV_COMBINE_WPH(DD, S)                                                               \
    switch (wph) {                                                                           \
    case 1: e = launch_pdl(piece_combine_kernel<DD, 1, S>, dim3(blocks), dim3(warps * 32), 0, \
                           stream, p); break;                                                \
    case 2: e = launch_pdl(piece_combine_kernel<DD, 2, S>, dim3(blocks), dim3(warps * 32), 0, \
                           stream, p); break;                                                \
    case 4: e = launch_pdl(piece_combine_kernel<DD, 4, S>, dim3(blocks), dim3(warps * 32), 0, \
                           stream, p); break;                                                \
    case 8: e = launch_pdl(piece_combine_kernel<DD, 8, S>, dim3(blocks), dim3(warps * 32), 0, \
                           stream, p); break;                                                \
    default: e = launch_pdl(piece_combine_kernel<DD, 16, S>, dim3(blocks), dim3(warps * 32), \
                            0, stream, p); break;                                            \
    }
    if (D == 64) {
        if (ds == 1) { PKV_COMBINE_WPH(64, 1) } else { PKV_COMBINE_WPH(64, 2) }
    } else {
        if (ds == 1) { PKV_COMBINE_WPH(128, 1) }
        else if (ds == 2) { PKV_COMBINE_WPH(128, 2) }
        else { PKV_COMBINE_WPH(128, 4) }
    }
#undef PKV_COMBINE_WPH
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace pkv
