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
// query heads (token-major) of one (row, kv head); query row t of a tile
// lives in lane t of tensor memory.  A unit is two consecutive tiles (A, B)
// whose keys stream in blocks of 128; one persistent block per SM walks a
// list of units:
//   - Q, K and V are loaded by TMA (3-D tiled tensor maps, 128-byte swizzle):
//     Q as one box per tile and 64 dims, K and V as one box per page and 64
//     dims; page sizes that are not a power of two >= 8 are gathered with
//     16-byte cp.async into the same swizzled layout;
//   - S = Q K^T (M 128, N 128, K = D in steps of 16) goes to tensor memory;
//   - a row's two threads each read half of its S (64 keys), mask keys past
//     its position, exchange their halves' max, update the fp32 online
//     softmax (log2 domain, the scale folded into one FFMA per exponent; l
//     from the fp32 terms at D = 128), rescale their halves of O in tensor
//     memory only when the max has grown by more than 2^8, and write P
//     (bf16) back over S;
//   - O += P V (M 128, N = D, K = 128) takes P from tensor memory and V
//     (MN-major) from shared memory; at D = 64 V has 16 more columns of
//     ones (N = 80), so the product also sums l;
//   - at a unit's end each thread loads its half row of O, hands O back,
//     and its lane group stores the rows in whole runs;
//   - tile A's products are issued by one thread and tile B's by another,
//     taking turns one run at a time, so each makes its waits and commits
//     while the other's run goes out.
// With a workspace (paged_prefill_attn_ws), a list whose last round would
// leave at least half the SMs idle cuts that round's units along their key
// blocks (the split-KV of the decode, applied to prefill): each part stores
// its rows normalised on its own base, with the rows' (base, l), in a
// workspace slot, and prefill_merge_kernel combines the parts.
// Every mbarrier wait is time-bounded; tensor memory is allocated at the
// start and released on every path.
#include <cmath>
#include <cudaTypedefs.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr unsigned kAllTc = 0xffffffffu;
// the position of a softmax row with no query: below every key
constexpr int kNoQuery = -(1 << 30);

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

// 32 consecutive fp32 columns of this thread's TMEM lane, load and wait in
// one asm statement.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31"
                 "}, [%32];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                 "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                 "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                 "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                 "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// One fp32 column of this thread's TMEM lane: load (and wait), store.
__device__ __forceinline__ float tmem_ld1(uint32_t taddr)
{
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r)
                 : "r"(taddr)
                 : "memory");
    return __uint_as_float(r);
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr),
                 "r"(__float_as_uint(v))
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
                 "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32"
                 "};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                 "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                 "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
                 "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                 "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                 "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
                 "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                 "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
                 "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])),
                 "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                 "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
                 "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
                 "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                 "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
}

__device__ __forceinline__ void tmem_st32w(uint32_t taddr, const uint32_t (&w)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
                 "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32"
                 "};" ::"r"(taddr),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]),
                 "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]), "r"(w[17]), "r"(w[18]),
                 "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]), "r"(w[24]),
                 "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]),
                 "r"(w[31])
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

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// cp.async completion of this thread's earlier copies arrives on bar (the
// barrier's count includes one arrival per loading thread).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// ---------------------------------------------------------------------------
// The kernel's layout.  Two query tiles (A, B) per block share every
// 128-key K/V block.  Tensor memory: S of tile x in columns
// [128 x, 128 x + 128), O of tile x at 256 + D x.  Each row's thread reads
// its row of S, runs its online softmax and writes P (bf16 pairs) back over
// the first 64 columns of its S; O += P V then takes P from tensor memory as
// the A operand (K-major: lane = query row, column c = keys 2c and 2c + 1)
// and V from shared memory, so the only shared-memory operands left are Q,
// K and V.  The MMA thread alternates the tiles:
//   P V of tile A (block j), S of tile A (block j + 1),
//   P V of tile B (block j), S of tile B (block j + 1),
// so while one tile's rows run their softmax the tensor cores work on the
// other tile.  A tile's next S overwrites the columns its P V reads; both are
// issued by one thread and the tensor cores run them in issue order.  The
// commit behind each S also covers the P V before it, so a softmax that sees
// its S may rescale O: no MMA touches that O until its next P arrives.
// K and V have rings of their own (K is needed one P V earlier than V).
template <int D>
struct PrefillCfg {
    static constexpr int kRows = 128;                      // query rows of one tile
    static constexpr int kKeys = 128;                      // keys of one K/V block
    static constexpr int kKStages = D <= 64 ? 4 : 2;
    static constexpr int kVStages = D <= 64 ? 4 : 3;
    // warps 0-7: softmax of tile A, 8-15: tile B (a row's two threads, in
    // warpgroups 2x and 2x + 1, take 64 of a block's 128 keys each); warp
    // 16: tensor-memory owner and tile A's products; warp 17: K loads; warp
    // 18: V and Q loads; warp 19: tile B's products
    static constexpr int kSoftmaxWarps = 16;
    static constexpr int kMmaWarp = kSoftmaxWarps;
    static constexpr int kMmaWarpB = 19;               // tile B's products
    static constexpr int kThreads = 20 * 32;
    // 20 warps leave a thread 96 registers (65,536 / 640, in steps of 8):
    // enough for a half row of S (64) in the softmax and for the other roles
    // a tile or block of 128 rows: D / 64 regions of 128 rows x 128 bytes
    // (64 dims each), 128-byte swizzled
    static constexpr int kRegionBytes = 128 * 128;
    static constexpr int kQBytes = D / 64 * kRegionBytes;  // one query tile
    static constexpr int kKVBytes = D / 64 * kRegionBytes; // one K or V block
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKVBytes;
    static constexpr int kBarOff = kVOff + kVStages * kKVBytes + (D <= 64 ? kRegionBytes : 0);
    // k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2], p_full[2],
    // o_full[2], o_empty[2], q_full[2], q_empty[2], drain, xch_bar[2], turn[2],
    // rec_full[4], rec_empty[4]
    static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 25;
    // a row's two halves exchange their max (and at the end their l) here:
    // [tile][half][row] floats, one buffer (which leaves room for the third V
    // stage at D = 128).  A half's next write is ordered after its partner's
    // read of the last value: within a unit by P -> next S (the issuing
    // thread waits for every warp's P before the S behind the next write);
    // the l after the last max by the wait for the unit's last P V; a new
    // unit's first max after the l by a wait for o_empty (every warp of the
    // tile has read its l and O)
    static constexpr int kXchOff = kBarOff + kNumBars * 8;
    static constexpr int kXchBytes = 2 * 2 * kRows * 4;
    static constexpr int kTmemSlot = kXchOff + kXchBytes;
    static constexpr int kAbortOff = kTmemSlot + 4;
    // a split list's entry of each tile, by unit parity: its slot when it is
    // a part of a split unit, else -1
    static constexpr int kPartSlotOff = kAbortOff + 4;
    // the unit of each round, published by the K warp for the other roles:
    // a ring of kRecs records of 16 ints
    static constexpr int kRecs = 4;
    static constexpr int kRecOff = kPartSlotOff + 16;
    static constexpr int kSmemBytes = kRecOff + kRecs * 16 * 4;
    static_assert(kSmemBytes <= 232448, "shared memory per block");
    // the block holds all of tensor memory: its shared memory keeps a second
    // block off the SM (whose allocation would wait for this one's release)
    static_assert(2 * (kSmemBytes + 1024) > 233472, "one block per SM");
    static constexpr uint32_t kTmemCols = 512;
    // At D = 64 the row sums l come from the tensor cores: V gets 16 more
    // columns, all ones (one shared 128-key region of ones after the V ring,
    // the descriptor's LBO reaching it from each slot), so P V writes
    // l = sum of the row's bf16 P into O's column D (kOnesL).  At D = 128
    // tensor memory has no room for them.
    static constexpr bool kOnesL = D <= 64;
    static constexpr int kON = kOnesL ? D + 16 : D;        // columns of a tile's O
    static constexpr int kOnesOff = kVOff + kVStages * kKVBytes;  // the ones region (16 KB at D = 64)
    static constexpr uint32_t kOCol = 256;                 // O of tile x at kOCol + kON x
};

// Shared-memory descriptor of a 128-byte-swizzled operand (layout type 2).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return smem_desc(addr, lbo, sbo) | ((uint64_t)2 << 61);
}

// One box of a 3-D tiled tensor map into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
                 "r"(smem_addr(bar))
                 : "memory");
}

// D += A B with A (M 128, K 16, bf16) in tensor memory.
__device__ __forceinline__ void umma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bd,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
                 "r"(tmem_a), "l"(bd), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two floats as one packed f32x2 operand.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// (y0, y1) = (a0, a1) * b + c, one packed FMA (b, c: f32x2 operands).
__device__ __forceinline__ void ffma2(float &y0, float &y1, float a0, float a1, uint64_t b,
                                      uint64_t c)
{
    asm("{\n .reg .b64 a, r;\n mov.b64 a, {%2, %3};\n fma.rn.f32x2 r, a, %4, %5;\n"
        " mov.b64 {%0, %1}, r;\n}"
        : "=f"(y0), "=f"(y1)
        : "f"(a0), "f"(a1), "l"(b), "l"(c));
}

// (a0, a1) += (b0, b1), one packed add.
__device__ __forceinline__ void fadd2(float &a0, float &a1, float b0, float b1)
{
    asm("{\n .reg .b64 a, b, r;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
        " add.rn.f32x2 r, a, b;\n mov.b64 {%0, %1}, r;\n}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

// 2^x on the special-function unit (the PTX approximate instruction; 0 for -inf).
__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One unit of work: query tiles tB = n_tiles - 1 - 2 pair (the most keys
// first) and tA = tB - 1 (-1: idle) of row b's chunk, with kv head g.
struct PrefillUnit {
    int b, g, q0, q_len, L, tA, tB, kv_end, pg0;
    int kb0, n_kb;                 // the key blocks [kb0, kb0 + n_kb) this entry runs
    // a part of a split unit: slot << 9 | parts << 4 | part; -1 for a whole unit
    int part_id;
    bool table_ok;
};

// Wait for phase `parity` of `bar`; false if the time limit ran out or
// another role aborted.  The abort flag is read only once the phase is not
// already complete: a role that fails stops producing, so every role's next
// wait that blocks sees the flag.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity,
                                                   volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return true;
}

__device__ __forceinline__ void st_global_v8(void *dst, const uint32_t (&w)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Each lane's N consecutive outputs of its row (dst, 16-byte aligned;
// nullptr: none), v x inv rounded to bf16, stored by the whole warp.  A
// lane's outputs are G = N / 16 pieces of 32 bytes; the G lanes of each
// group first trade pieces (a G x G transpose by XOR shuffles), so that
// lane j holds piece j of the group's G rows and each store instruction
// writes whole runs of N x 2 bytes: 32 / G runs per instruction instead of
// 32 scattered pieces, far fewer cache-line requests for the load/store
// unit, which the block's shared-memory traffic and barriers also use.  A
// piece is one 32-byte store when every dst is 32-byte aligned (wide), else
// two 16-byte stores.
template <int N>
__device__ __forceinline__ void store_rows_warp(__nv_bfloat16 *dst, const float (&v)[N], float inv,
                                                int lane, bool wide)
{
    constexpr int G = N / 16;
    uint32_t w[G][8];
#pragma unroll
    for (int c = 0; c < G; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[c][i] = pack_bf16x2(v[16 * c + 2 * i] * inv, v[16 * c + 2 * i + 1] * inv);
    const int j = lane & (G - 1);
#pragma unroll
    for (int s = 1; s < G; s <<= 1) {
        const bool hi = (j & s) != 0;
#pragma unroll
        for (int c = 0; c < G; ++c) {
            if (c & s)
                continue;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t got = __shfl_xor_sync(kAllTc, hi ? w[c][i] : w[c | s][i], s);
                if (hi)
                    w[c][i] = got;
                else
                    w[c | s][i] = got;
            }
        }
    }
    const unsigned long long mine = reinterpret_cast<unsigned long long>(dst);
    const int b = lane & ~(G - 1);
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const unsigned long long row = __shfl_sync(kAllTc, mine, b + k);
        uint32_t *piece = reinterpret_cast<uint32_t *>(row) + 8 * j;
        if (row != 0ull) {
            if (wide) {
                st_global_v8(piece, w[k]);
            } else {
                *reinterpret_cast<uint4 *>(piece) = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
                *reinterpret_cast<uint4 *>(piece + 4) =
                    make_uint4(w[k][4], w[k][5], w[k][6], w[k][7]);
            }
        }
    }
}

// Unit u of the list: rows (b x Hkv + g) in groups of p.group_rows, the
// groups one after another and each group pair-major (its rows' largest
// pairs first); false when the unit has no work: a pair past its row's
// chunk, or a refused row.  flag: report refusals in the status.
__device__ __forceinline__ bool prefill_whole_unit(const PrefillParams &p, int u, PrefillUnit &w,
                                                   bool flag)
{
    const int rows = p.B * p.Hkv;
    int pair, rh;
    if (p.group_rows >= rows) {                        // one group: pair-major
        pair = u / rows;
        rh = u - pair * rows;
    } else {
        const int per_group = p.group_rows * p.pairs;
        const int grp = u / per_group, ul = u - grp * per_group;
        const int g_rows = min(p.group_rows, rows - grp * p.group_rows);
        pair = ul / g_rows;
        rh = grp * p.group_rows + (ul - pair * g_rows);
    }
    w.b = rh / p.Hkv;
    w.g = rh - w.b * p.Hkv;
    w.q0 = p.qo_indptr[w.b];
    const int q1 = p.qo_indptr[w.b + 1];
    w.L = p.seq_lens[w.b];
    const int k0 = p.kv_indptr[w.b], k1 = p.kv_indptr[w.b + 1];
    w.q_len = q1 - w.q0;
    const bool row_ok = w.q_len >= 0 && w.q0 >= 0 && q1 <= p.total_q && w.L >= 0 &&
                        w.L <= p.max_seq_len && w.q_len <= w.L;
    const bool first = flag && pair == 0 && w.g == 0;  // one report per row
    if (!row_ok) {
        if (first)
            tc_flag(p.status, kFlagBadLen);
        return false;
    }
    const int n_tiles = (w.q_len + p.tq - 1) / p.tq;
    if (first && (n_tiles + 1) / 2 > p.pairs)
        tc_flag(p.status, kFlagBadLen);                // chunk longer than max_q_len
    w.tB = n_tiles - 1 - 2 * pair;
    if (w.tB < 0)
        return false;
    w.tA = w.tB - 1;
    w.kv_end = w.L - w.q_len + min(w.q_len, (w.tB + 1) * p.tq);
    w.n_kb = (w.kv_end + 127) / 128;
    w.kb0 = 0;
    w.part_id = -1;
    w.pg0 = k0;
    const int npg = k1 - k0;
    w.table_ok = k0 >= 0 && npg >= 0 && k1 <= p.num_indices &&
                 (long long)npg * p.page_size >= (long long)w.L;
    if (!w.table_ok && flag)
        tc_flag(p.status, kFlagBadPage);
    return true;
}

// Entry u of the list: unit u, or in a list with a key split (kSplit), from
// p.split_base on, parts, p.split to a unit: part k of a unit of n blocks in
// np = min(p.split, n / kPrefillMinPartBlocks) parts (at least one) takes
// blocks [k n / np, (k + 1) n / np); false when the entry has no work (also
// a part past its unit's share).
template <bool kSplit>
__device__ __forceinline__ bool prefill_unit(const PrefillParams &p, int u, PrefillUnit &w,
                                             bool flag)
{
    if (kSplit && u >= p.split_base) {
        const int slot = u - p.split_base, part = slot % p.split;
        if (!prefill_whole_unit(p, p.split_base + slot / p.split, w, flag && part == 0))
            return false;
        const int np = max(1, min(p.split, w.n_kb / kPrefillMinPartBlocks));
        if (part >= np)
            return false;
        const int lo = part * w.n_kb / np, hi = (part + 1) * w.n_kb / np;
        w.kb0 = lo;
        w.n_kb = hi - lo;
        if (np > 1)
            w.part_id = slot << 9 | np << 4 | part;
        return true;
    }
    return prefill_whole_unit(p, u, w, flag);
}

// A unit as a ring record: [0] has work, then its fields.
__device__ __forceinline__ void unit_to_rec(int *rec, bool have, const PrefillUnit &w)
{
    rec[0] = have ? 1 : 0;
    rec[1] = w.b;
    rec[2] = w.g;
    rec[3] = w.q0;
    rec[4] = w.q_len;
    rec[5] = w.L;
    rec[6] = w.tA;
    rec[7] = w.tB;
    rec[8] = w.kv_end;
    rec[9] = w.pg0;
    rec[10] = w.kb0;
    rec[11] = w.n_kb;
    rec[12] = w.part_id;
    rec[13] = w.table_ok ? 1 : 0;
}

__device__ __forceinline__ bool rec_to_unit(const int *rec, PrefillUnit &w)
{
    w.b = rec[1];
    w.g = rec[2];
    w.q0 = rec[3];
    w.q_len = rec[4];
    w.L = rec[5];
    w.tA = rec[6];
    w.tB = rec[7];
    w.kv_end = rec[8];
    w.pg0 = rec[9];
    w.kb0 = rec[10];
    w.n_kb = rec[11];
    w.part_id = rec[12];
    w.table_ok = rec[13] != 0;
    return rec[0] != 0;
}

// A persistent block (one per SM) takes one unit per round of gridDim.x
// units; every role walks the same list and keeps its ring and phase
// counters across units, so one unit's epilogue overlaps the next unit's
// loads and first products.
// kSplit: the list ends in a key split's parts (p.split > 1); without one the
// kernel has no trace of it (every entry a whole unit from key 0).
template <int D, bool kSplit>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p)
{
    using C = PrefillCfg<D>;
    constexpr int CH = D / 8;                      // 16-byte chunks per row
    constexpr int KS = C::kKStages, VS = C::kVStages;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *k_full = bars, *k_empty = k_full + KS;
    uint64_t *v_full = k_empty + KS, *v_empty = v_full + VS;
    uint64_t *s_full = v_empty + VS, *p_full = s_full + 2, *o_full = p_full + 2;
    uint64_t *o_empty = o_full + 2, *q_full = o_empty + 2, *q_empty = q_full + 2;
    uint64_t *drain = q_empty + 2, *xch_bar = drain + 1, *turn = xch_bar + 2;
    uint64_t *rec_full = turn + 2, *rec_empty = rec_full + C::kRecs;
    int *recs = reinterpret_cast<int *>(smem + C::kRecOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kAbortOff);
    volatile int *part_slot = reinterpret_cast<volatile int *>(smem + C::kPartSlotOff);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_rep = p.n_rep, tq = p.tq;
    const int rows_used = tq * n_rep;
    const int n_units = p.n_units;
    // round r's unit of this block: the rounds run the list alternately
    // forwards and backwards over the blocks, so a block with a large unit
    // in one round gets a small one in the next
    auto unit_index = [&](int r) {
        const int G = (int)gridDim.x, c = (int)blockIdx.x;
        return r * G + ((r & 1) ? G - 1 - c : c);
    };
    // round r's unit as the K warp published it (false: the wait gave up)
    auto take_unit = [&](int r, PrefillUnit &w, bool &have) {
        if (!mbar_wait_or_abort(&rec_full[r % C::kRecs], (uint32_t)((r / C::kRecs) & 1),
                                abort_flag))
            return false;
        have = rec_to_unit(recs + (r % C::kRecs) * 16, w);
        return true;
    };

    if (tid == 0) {
        for (int s = 0; s < KS; ++s) {
            mbar_init(&k_full[s], 32);                 // the K warp's lanes
            mbar_init(&k_empty[s], 2);                 // both tiles' S
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(&v_full[s], 32);                 // the V warp's lanes
            mbar_init(&v_empty[s], 2);                 // both tiles' P V
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 8);                  // the tile's 8 softmax warps
            mbar_init(&o_full[x], 1);
            mbar_init(&o_empty[x], 8);                 // the tile's epilogue has read O
            mbar_init(&xch_bar[x], 8);                 // a block's halves exchanged
            mbar_init(&q_full[x], 32);                 // the V warp's lanes
            mbar_init(&q_empty[x], 1);                 // the unit's last S has read Q
        }
        mbar_init(drain, 2);                           // both issuing threads
        mbar_init(&turn[0], 1);
        mbar_init(&turn[1], 1);
        mbar_arrive(&turn[0]);                         // tile A's run goes first
        for (int i = 0; i < C::kRecs; ++i) {
            mbar_init(&rec_full[i], 1);                // the K warp wrote the record
            // every reader: the V warp, both issuing threads, 16 softmax warps
            mbar_init(&rec_empty[i], 1 + 2 + C::kSoftmaxWarps);
        }
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
    if constexpr (C::kOnesL) {
        // bf16 1.0 in every column of the ones region (whatever the swizzle,
        // each of the 16 columns the products read is 1), for the tensor cores
        uint4 *ones = reinterpret_cast<uint4 *>(smem + C::kOnesOff);
        for (int i = tid; i < C::kRegionBytes / 16; i += C::kThreads)
            ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        fence_proxy_async_smem();
    }
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&]() {
        *abort_flag = 1;
        tc_flag(p.status, kFlagTimeout);
    };

    if (warp >= C::kMmaWarp) {
        if (warp == C::kMmaWarp + 1 || warp == C::kMmaWarp + 2) {
            // ====================== K/V loads ===================================
            // warp 17 fills the K ring, warp 18 the V ring.  A slot holds a block's
            // 128 keys as D / 64 regions of 128 rows x 128 bytes (64 dims of a
            // key), 128-byte swizzled: 16-byte chunk c of row r at c ^ (r & 7).
            const bool is_v = warp == C::kMmaWarp + 2;
            const int ns = is_v ? VS : KS;
            uint64_t *full = is_v ? v_full : k_full;
            uint64_t *empty = is_v ? v_empty : k_empty;
            const uint32_t ring = sbase + (is_v ? C::kVOff : C::kKOff);
            const __nv_bfloat16 *pool = is_v ? p.v_pool : p.k_pool;
            const CUtensorMap *tmap = is_v ? &p.tmap_v : &p.tmap_k;
            // cp.async: one instruction copies chunks [4 cq, 4 cq + 4) of 8
            // keys, lane = key (lane & 7), chunk 4 cq + (lane >> 3): each key's
            // 64 bytes are two whole L2 sectors, and the swizzle spreads the 8
            // rows' chunks over all banks
            const int kl = lane & 7, cl = lane >> 3;
            int kb = 0;                                    // blocks issued, over all units
            int qit = 0;                                   // units whose Q the V warp loaded
            for (int r = 0; r * (int)gridDim.x < n_units && !*abort_flag; ++r) {
                PrefillUnit w;
                bool have = false;
                if (!is_v) {
                    // the K warp looks the unit up (reporting refusals once)
                    // and publishes it for the other roles
                    const int u = unit_index(r);
                    have = u < n_units && prefill_unit<kSplit>(p, u, w, lane == 0);
                    if (lane == 0) {
                        const bool free_slot =
                            r < C::kRecs ||
                            mbar_wait_or_abort(&rec_empty[r % C::kRecs],
                                               (uint32_t)((r / C::kRecs - 1) & 1), abort_flag);
                        if (free_slot) {
                            unit_to_rec(recs + (r % C::kRecs) * 16, have, w);
                            mbar_arrive(&rec_full[r % C::kRecs]);
                        } else {
                            fail();
                        }
                    }
                    __syncwarp();
                } else {
                    const bool got = __all_sync(kAllTc, take_unit(r, w, have));
                    __syncwarp();
                    if (lane == 0 && got)
                        mbar_arrive(&rec_empty[r % C::kRecs]);
                    if (!got) {
                        if (lane == 0)
                            fail();
                        break;
                    }
                }
                if (!have)
                    continue;
                // the V warp also loads the unit's Q (row m = token m / n_rep,
                // head m % n_rep, swizzled like K), each tile's once the previous
                // unit's last S of that tile has read it, before the unit's V;
                // an idle tile A is not loaded (its rows are masked out whatever
                // they hold)
                for (int x = 0; x < 2 && is_v && !*abort_flag; ++x) {
                    if (qit > 0 &&
                        !mbar_wait_bounded(&q_empty[x], (uint32_t)((qit - 1) & 1))) {
                        if (lane == 0)
                            fail();
                        break;
                    }
                    const int t = x == 0 ? w.tA : w.tB;
                    const uint32_t dst = sbase + x * C::kQBytes;
                    if (p.q_tma) {
                        const uint32_t bytes = t >= 0 ? (uint32_t)((D / 64) * rows_used * 128) : 0u;
                        if (lane == 0)
                            mbar_arrive_expect_tx(&q_full[x], bytes);
                        else
                            mbar_arrive(&q_full[x]);
                        __syncwarp();
                        if (t >= 0 && lane < D / 64)
                            tma_load_3d(dst + lane * C::kRegionBytes, &p.tmap_q, 64 * lane,
                                        w.g * n_rep, w.q0 + t * tq, &q_full[x]);
                    } else {
                        for (int e = lane; e < C::kRows * CH; e += 32) {
                            const int m = e / CH, c = e % CH;
                            const int tok = m / n_rep, hq = m - tok * n_rep;
                            const bool live = t >= 0 && m < rows_used && tok < w.q_len - t * tq;
                            const __nv_bfloat16 *src =
                                live ? p.q + ((size_t)(w.q0 + t * tq + tok) * p.Hq +
                                              (size_t)w.g * n_rep + hq) * D + c * 8
                                     : p.q;
                            cp_async16(dst + (c >> 3) * C::kRegionBytes + m * 128 +
                                           (((c & 7) ^ (m & 7)) << 4),
                                       src, live ? 16u : 0u);
                        }
                        cp_async_arrive(&q_full[x]);
                    }
                }
                if (is_v)
                    ++qit;
                for (int j = 0; j < w.n_kb; ++j) {
                    const int slot = kb % ns;
                    if (kb >= ns) {
                        if (!mbar_wait_bounded(&empty[slot], (uint32_t)(((kb / ns) - 1) & 1)) &&
                            lane == 0)
                            fail();
                        __syncwarp();
                    }
                    if (*abort_flag)
                        break;
                    const uint32_t dst = ring + slot * C::kKVBytes;
                    const int key0 = (w.kb0 + j) * C::kKeys;
                    const int nkeys = min(C::kKeys, w.kv_end - key0);
                    // K rows past kv_end are masked out of S whatever they hold,
                    // so a K block loads whole boxes; V rows past it meet P = 0 and
                    // must be finite, so a partial V block is copied with zero fill
                    if (p.use_tma && (!is_v || nkeys == C::kKeys)) {
                        const int R = p.tma_rows;
                        const int nbox = (nkeys + R - 1) / R;
                        if (lane == 0)
                            mbar_arrive_expect_tx(&full[slot],
                                                  (uint32_t)(nbox * (D / 64) * R * 128));
                        else
                            mbar_arrive(&full[slot]);
                        __syncwarp();
                        for (int bx = lane; bx < nbox; bx += 32) {
                            const int tok = key0 + bx * R;
                            const int pi = tok >> p.ps_shift;
                            int page = w.table_ok ? __ldg(p.kv_indices + w.pg0 + pi) : 0;
                            if (page < 0 || page >= p.num_pages) {
                                tc_flag(p.status, kFlagBadPage);
                                page = 0;
                            }
                            const int row = (page << p.ps_shift) + (tok - (pi << p.ps_shift));
#pragma unroll
                            for (int h = 0; h < D / 64; ++h)
                                tma_load_3d(dst + h * C::kRegionBytes + bx * R * 128, tmap, 64 * h,
                                            w.g, row, &full[slot]);
                        }
                    } else {
                        size_t offs[C::kKeys / 8];
                        unsigned live = 0u;
#pragma unroll
                        for (int kg = 0; kg < C::kKeys / 8; ++kg) {
                            const int tok = key0 + kg * 8 + kl;
                            offs[kg] = 0;
                            if (tok < w.kv_end) {
                                const int pi =
                                    p.ps_shift >= 0 ? (tok >> p.ps_shift) : (tok / p.page_size);
                                const int sl = tok - pi * p.page_size;
                                int page = w.table_ok ? __ldg(p.kv_indices + w.pg0 + pi) : 0;
                                if (page < 0 || page >= p.num_pages) {
                                    tc_flag(p.status, kFlagBadPage);
                                    page = 0;
                                }
                                offs[kg] = (((size_t)page * p.page_size + sl) * p.Hkv + w.g) * D;
                                live |= 1u << kg;
                            }
                        }
#pragma unroll
                        for (int kg = 0; kg < C::kKeys / 8; ++kg) {
                            const uint32_t row = dst + (kg * 8 + kl) * 128;
#pragma unroll
                            for (int cq = 0; cq < CH / 4; ++cq) {
                                const int c = 4 * cq + cl;
                                cp_async16(row + (c >> 3) * C::kRegionBytes + (((c & 7) ^ kl) << 4),
                                           pool + offs[kg] + c * 8, ((live >> kg) & 1u) ? 16u : 0u);
                            }
                        }
                        cp_async_arrive(&full[slot]);
                    }
                    ++kb;
                }
            }
            cp_async_wait_all();
            // the block exits only after its copies land: after an abort the MMA
            // thread may not have waited for the last slots issued
            for (int k = max(0, kb - ns); k < kb; ++k)
                (void)mbar_wait_bounded(&full[k % ns], (uint32_t)((k / ns) & 1));
            if (is_v && qit > 0)
                for (int x = 0; x < 2; ++x)
                    (void)mbar_wait_bounded(&q_full[x], (uint32_t)((qit - 1) & 1));
        } else {
            // ====================== tensor-core issue ===========================
            // warp 16 issues tile A's products, warp 19 tile B's.  They take
            // turns, one run each (the S of a unit's first block; then P V of
            // block j with S of block j + 1), in the order one thread would
            // issue them.  Each thread waits for its next run's data and P, and
            // makes its commits, while the other's run goes out, so the tensor
            // cores always have a run queued.
            const int x = warp == C::kMmaWarpB ? 1 : 0;
            constexpr uint32_t kIdescS = instr_desc(128, C::kKeys, 0);
            constexpr uint32_t kIdescO = instr_desc(128, C::kON, 1);
            // Q and K: 128-byte swizzle, K-major: 8-row groups 1 KB apart (SBO),
            // a 16-dim step 32 bytes into the row, the next 64 dims in the next
            // region.  V: 128-byte swizzle, MN-major: 64-dim atoms one region
            // apart (LBO), 8-key groups 1 KB apart (SBO); at D = 64 one atom spans
            // N, so LBO is unused (1 KB keeps every address inside the slot
            // however it were read).
            const uint64_t dq = smem_desc_sw128(sbase, 16, 1024);
            const uint64_t dk = smem_desc_sw128(sbase + C::kKOff, 16, 1024);
            const uint64_t dv =
                smem_desc_sw128(sbase + C::kVOff, D > 64 ? C::kRegionBytes : 1024, 1024);
            if (lane == 0) {
                bool ok = true;
                auto wait_only = [&](uint64_t *bar, uint32_t parity) {
                    ok = ok && mbar_wait_or_abort(bar, parity, abort_flag);
                    return ok;
                };
                const bool k_generic = !p.use_tma;
                // Q and K share the swizzled K-major form: step s is 32 bytes into
                // region s / 4
                const uint64_t dq_x = dq + (uint64_t)((x * C::kQBytes) >> 4);
                auto issue_s = [&](int kslot) {
                    const uint64_t dk_s = dk + (uint64_t)((kslot * C::kKVBytes) >> 4);
#pragma unroll
                    for (int s = 0; s < D / 16; ++s) {
                        const uint64_t ks =
                            (uint64_t)(((s >> 2) * C::kRegionBytes + (s & 3) * 32) >> 4);
                        umma(tmem + 128 * x, dq_x + ks, dk_s + ks, kIdescS, s > 0);
                    }
                };
                auto issue_pv = [&](int vslot, bool first) {
                    // at D = 64 the second 64-column atom of V (its columns 64..79:
                    // ones) is the ones region, LBO bytes on from the slot
                    const uint64_t dv_s =
                        C::kOnesL ? smem_desc_sw128(sbase + C::kVOff + vslot * C::kKVBytes,
                                                    C::kOnesOff - C::kVOff - vslot * C::kKVBytes,
                                                    1024)
                                  : dv + (uint64_t)((vslot * C::kKVBytes) >> 4);
#pragma unroll
                    for (int s = 0; s < C::kKeys / 16; ++s)
                        umma_ta(tmem + C::kOCol + C::kON * x, tmem + 128 * x + 8 * s,
                                dv_s + (uint64_t)((s * 16 * 128) >> 4), kIdescO,
                                (!first || s > 0) ? 1u : 0u);
                };
                // the turn: this tile's run of products goes out once the other
                // tile's run has been issued, then passes the turn back
                uint32_t turns = 0u;
                auto take_turn = [&]() {
                    ok = ok && mbar_wait_or_abort(&turn[x], turns & 1u, abort_flag);
                    ++turns;
                    if (ok)
                        tc_fence_after();
                    return ok;
                };
                auto pass_turn = [&]() { mbar_arrive(&turn[x ^ 1]); };
                int kb = 0, it = 0;                        // blocks and units consumed
                uint32_t pc = 0u;                          // P hand-offs consumed
                for (int r = 0; r * (int)gridDim.x < n_units && ok; ++r) {
                    // round r's unit from the K warp's record
                    const int rs = r % C::kRecs;
                    const int *rec = recs + rs * 16;
                    if (!wait_only(&rec_full[rs], (uint32_t)((r / C::kRecs) & 1)))
                        break;
                    const bool have = rec[0] != 0;
                    PrefillUnit w;
                    w.kv_end = rec[8];
                    w.kb0 = rec[10];
                    w.n_kb = rec[11];
                    mbar_arrive(&rec_empty[rs]);
                    if (!have)
                        continue;
                    const int n_kb = w.n_kb;
                    if (!wait_only(&q_full[x], (uint32_t)(it & 1)) ||
                        !wait_only(&k_full[kb % KS], (uint32_t)((kb / KS) & 1)))
                        break;
                    // stages filled by cp.async: their generic-proxy writes
                    // before the tensor cores' reads
                    if (!p.q_tma || k_generic)
                        fence_proxy_async_smem();
                    // S of block 0 (the tile's last S of the previous unit was
                    // issued before its P V, so these columns are free in order)
                    if (!take_turn())
                        break;
                    issue_s(kb % KS);
                    pass_turn();
                    umma_commit(&s_full[x]);
                    if (n_kb == 1)
                        umma_commit(&q_empty[x]);
                    umma_commit(&k_empty[kb % KS]);
                    for (int j = 0; j < n_kb && ok; ++j) {
                        const int kj = kb + j;
                        const bool more = j + 1 < n_kb;
                        // this run's data and P, waited for while the other
                        // tile's run is issued
                        const bool v_gen =
                            !p.use_tma || w.kv_end - (w.kb0 + j) * C::kKeys < C::kKeys;
                        if (!wait_only(&v_full[kj % VS], (uint32_t)((kj / VS) & 1)))
                            break;
                        if (more &&
                            !wait_only(&k_full[(kj + 1) % KS], (uint32_t)(((kj + 1) / KS) & 1)))
                            break;
                        if (v_gen || (more && k_generic))
                            fence_proxy_async_smem();
                        if (!wait_only(&p_full[x], pc & 1u))
                            break;
                        ++pc;
                        // the unit's first P V overwrites O: the previous unit's
                        // epilogue must have read it
                        if (j == 0 && it > 0 && !wait_only(&o_empty[x], (uint32_t)((it - 1) & 1)))
                            break;
                        if (!take_turn())
                            break;
                        issue_pv(kj % VS, j == 0);
                        if (more)
                            issue_s((kj + 1) % KS);
                        pass_turn();
                        umma_commit(&v_empty[kj % VS]);
                        if (more) {
                            umma_commit(&s_full[x]);
                            if (j + 2 == n_kb)
                                umma_commit(&q_empty[x]);
                            umma_commit(&k_empty[(kj + 1) % KS]);
                        } else {
                            umma_commit(&o_full[x]);
                        }
                    }
                    kb += n_kb;
                    ++it;
                }
                if (!ok)
                    fail();
                // tracks every product this thread issued: tensor memory is
                // released only after both threads' products are done
                umma_commit(drain);
            }
            __syncwarp();
        }
    } else {
        // ====================== softmax of tile x, row m, half h ============
        // warps 0-7 run tile A, 8-15 tile B; warpgroup h of a tile takes keys
        // [64 h, 64 h + 64) of each 128-key block, so a row's two threads
        // (one tensor-memory lane) each handle half of its keys.  Per block
        // they exchange their halves' max through shared memory (one buffer,
        // one mbarrier phase per block and tile), keep their own part of l
        // (at D = 128), and each rescales and stores its D / 2 columns of O.
        // The hand-offs to the MMA thread take one arrival per warp.
        const int x = warp >> 3, h = (warp >> 2) & 1;
        const int m = tid & (C::kRows - 1);
        const int tok_m = m / n_rep;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + 128 * x + lane_off;
        const uint32_t t_o = tmem + C::kOCol + C::kON * x + (D / 2) * h + lane_off;
        const uint32_t t_l = tmem + C::kOCol + C::kON * x + D + lane_off;  // kOnesL: l
        float *xch = reinterpret_cast<float *>(smem + C::kXchOff) + x * 2 * C::kRows;
        const float sl2 = p.scale_log2;
        bool ok = true;
        auto timed_out = [&]() {
            ok = false;
            if (lane == 0)
                fail();
        };
        uint32_t sc = 0u;                              // S hand-offs consumed
        uint32_t xc = 0u;                              // exchanges done
        // publish v as this half's value of exchange xc and return the other
        // half's (false: the wait timed out).  The tensor-memory fences order
        // each half's reads of S before the other half's P overwrites them.
        auto exchange = [&](float v, float &other) {
            float *buf = xch;
            buf[h * C::kRows + m] = v;
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&xch_bar[x]);
            const bool got = mbar_wait_or_abort(&xch_bar[x], xc & 1u, abort_flag);
            tc_fence_after();
            ++xc;
            other = buf[(h ^ 1) * C::kRows + m];
            return got;
        };
        int it = 0;
        for (int r = 0; r * (int)gridDim.x < n_units && ok; ++r) {
            // round r's unit from the K warp's record, each field read where
            // it is used (the slot is released after the epilogue)
            const int rs = r % C::kRecs;
            const int *rec = recs + rs * 16;
            ok = mbar_wait_or_abort(&rec_full[rs], (uint32_t)((r / C::kRecs) & 1), abort_flag);
            if (!__all_sync(kAllTc, ok)) {
                timed_out();
                break;
            }
            auto release = [&]() {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&rec_empty[rs]);
            };
            if (rec[0] == 0) {
                release();
                continue;
            }
            if (kSplit && m == 0 && h == 0)
                part_slot[2 * x + (it & 1)] = rec[12] >= 0 ? rec[12] >> 9 : -1;
            const int t = rec[x == 0 ? 6 : 7];
            const int q_len = rec[4];
            const int ntok = t >= 0 ? min(tq, q_len - t * tq) : 0;
            // positions counted from the entry's first key (a part of a split
            // unit starts at block kb0); a row with no query masks every key
            const int pos_first = rec[5] - q_len + (t >= 0 ? t * tq : 0) - rec[10] * C::kKeys;
            const int pos =
                (t >= 0 && m < rows_used && tok_m < ntok) ? pos_first + tok_m : kNoQuery;
            float m_run = -INFINITY, l_run = 0.f;
            const int n_kb = rec[11];
            // the partner half has read the previous unit's l (it loaded O
            // after it) before this unit's first max overwrites it
            if (!C::kOnesL && it > 0) {
                ok = mbar_wait_or_abort(&o_empty[x], (uint32_t)((it - 1) & 1), abort_flag);
                if (!__all_sync(kAllTc, ok)) {
                    timed_out();
                    break;
                }
            }
            for (int j = 0; j < n_kb; ++j) {
                ok = mbar_wait_or_abort(&s_full[x], sc & 1u, abort_flag);
                ++sc;
                if (!__all_sync(kAllTc, ok)) {
                    timed_out();
                    break;
                }
                tc_fence_after();
                float sv[64];
                tmem_ld64(t_s + 64 * h, sv);
                const int key0 = j * C::kKeys + 64 * h;
                if (key0 + 63 > pos_first) {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        sv[i] = key0 + i > pos ? -INFINITY : sv[i];
                }
                // this half's max: three-input max over 8 independent chains
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    mx8[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
                for (int k = 1; k < 4; ++k)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mx8[i] = fmax3(mx8[i], sv[16 * k + i], sv[16 * k + 8 + i]);
                const float mh = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                // the row's max from both halves (both threads of the row
                // then take the same decisions below)
                float mo;
                ok = exchange(mh, mo);
                if (!__all_sync(kAllTc, ok)) {
                    timed_out();
                    break;
                }
                const float mx = fmaxf(mh, mo) * sl2;
                // a new base only when the max grows by more than 2^8 (or first)
                const bool rebase = mx > m_run + 8.f;
                float alpha = 1.f;
                if (rebase) {
                    alpha = ex2_fast(m_run - mx);      // 0 while m_run is -inf
                    m_run = mx;
                    if constexpr (!C::kOnesL)
                        l_run *= alpha;
                }
                const float nbase = m_run == -INFINITY ? 0.f : -m_run;
                const uint64_t scale2 = f32x2(sl2, sl2), base2 = f32x2(nbase, nbase);
                float ls[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    ls[i] = 0.f;
                // P of this half's keys over columns [32 h, 32 h + 32) of S
                // (the other half's S there was read before the exchange);
                // the exponent's argument and l (from the fp32 terms) as
                // packed pairs
                uint32_t pw[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float y0, y1;
                    ffma2(y0, y1, sv[2 * i], sv[2 * i + 1], scale2, base2);
                    const float e0 = ex2_fast(y0), e1 = ex2_fast(y1);
                    pw[i] = pack_bf16x2(e0, e1);
                    if constexpr (!C::kOnesL)       // at D = 64 P V sums l
                        fadd2(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], e0, e1);
                }
                tmem_st32w(t_s + 32 * h, pw);
                if constexpr (!C::kOnesL)
                    l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) +
                             ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                // O is quiescent here: the commit behind this S covered the
                // last P V, and the next one waits for this P
                if (__any_sync(kAllTc, rebase && j > 0)) {
#pragma unroll 1
                    for (int c0 = 0; c0 < D / 2; c0 += 32) {
                        float v[32];
                        tmem_ld32(t_o + c0, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] *= alpha;
                        tmem_st32(t_o + c0, v);
                    }
                    if (C::kOnesL && h == 1)          // l, O's column D, once
                        tmem_st1(t_l, tmem_ld1(t_l) * alpha);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[x]);
            }
            if (!ok)
                break;
            // ---- normalise and store this tile's rows; then O is free ------
            // the last P V done (every warp's last P, so the partner's read of
            // the last max, came before it), then the halves' l
            ok = mbar_wait_or_abort(&o_full[x], (uint32_t)(it & 1), abort_flag);
            float lo = 0.f;
            if constexpr (!C::kOnesL)
                ok = ok && exchange(l_run, lo);
            if (!__all_sync(kAllTc, ok)) {
                timed_out();
                break;
            }
            tc_fence_after();
            // this thread's D / 2 columns of O and the row's l (both halves'
            // sums, or at D = 64 O's column D) into registers: O is then
            // free.  Its hand-off and the record's release go before the
            // row's stores, since an arrival orders the thread's earlier
            // global stores and would wait for them to complete.
            const float l_row = C::kOnesL ? tmem_ld1(t_l) : l_run + lo;
            float ov[D / 2];
            if constexpr (D / 2 == 64)
                tmem_ld64(t_o, ov);
            else
                tmem_ld32(t_o, ov);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&o_empty[x]);
            // a part of a split unit stores its rows like any entry, into its
            // workspace slot, with the row's (base, l) beside them for the
            // merge kernel (its slot was published at the unit's start; the
            // max exchange of every block since orders that write before
            // this read)
            __nv_bfloat16 *orow = nullptr;
            float2 *mlrow = nullptr;
            const int slot = kSplit ? part_slot[2 * x + (it & 1)] : -1;
            if (slot >= 0) {
                const size_t tile = (size_t)slot * 2 + x;
                orow = p.ws_o + (tile * C::kRows + m) * D + (D / 2) * h;
                if (h == 0)
                    mlrow = p.ws_ml + tile * C::kRows + m;
            } else if (pos != kNoQuery) {
                const int hh = m - tok_m * n_rep;
                orow = p.out +
                       ((size_t)(rec[3] + t * tq + tok_m) * p.Hq + (size_t)rec[2] * n_rep + hh) * D +
                       (D / 2) * h;
            }
            release();
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            if (mlrow != nullptr)
                *mlrow = make_float2(m_run, l_row);
            // whole runs, by 32-byte stores where the output allows them
            // (the workspace always does)
            store_rows_warp<D / 2>(orow, ov, inv, lane, slot >= 0 || p.out_align32);
            ++it;
        }
    }
    // every role is done; on an abort the MMA warp waits (bounded) for the
    // tensor cores to drain before tensor memory is released
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        if (lane == 0)
            (void)mbar_wait_bounded(drain, 0u);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(C::kTmemCols)
                     : "memory");
    }
}

// The key split's merge: D / 8 blocks per split unit and tile, a thread per
// (row, 16-byte column group); units of the split round that were not cut
// wrote their outputs themselves.  Each part left its rows normalised on a
// base of its own with (base, l): part i weighs l_i 2^(base_i - the largest
// base), and the parts are summed in part order (the pages' split-KV merge
// by (max, sum), as decode_combine does per split).
template <int D>
__global__ void __launch_bounds__(128) prefill_merge_kernel(const __grid_constant__ PrefillParams p)
{
    using C = PrefillCfg<D>;
    constexpr int kGroups = D / 8;                     // 16-byte column groups per row
    const int blk = (int)blockIdx.x / kGroups, sub = (int)blockIdx.x - blk * kGroups;
    const int su = blk >> 1, x = blk & 1;
    const int e = sub * (int)blockDim.x + (int)threadIdx.x;   // (row, group) of the tile
    const int m = e / kGroups, c = (e - m * kGroups) * 8;
    const size_t tile0 = (size_t)su * p.split * 2 + x;    // part i: tile0 + 2 i
    grid_dependency_wait();
    // the first four parts' rows load while the unit is looked up (every
    // unit of the split round owns p.split slots, written or not)
    float2 ml[4];
    uint4 a[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const size_t tile = tile0 + 2 * (size_t)(j < p.split ? j : 0);
        ml[j] = __ldcg(&p.ws_ml[tile * C::kRows + m]);
        a[j] = __ldcg(reinterpret_cast<const uint4 *>(p.ws_o + (tile * C::kRows + m) * D + c));
    }
    PrefillUnit w;
    // the unit as its first part sees it: np parts, or not cut
    if (!prefill_unit<true>(p, p.split_base + su * p.split, w, false) || w.part_id < 0)
        return;                                        // no work, or written whole
    const int np = (w.part_id >> 4) & 31;
    const int t = x == 0 ? w.tA : w.tB;
    const int n_rep = p.n_rep, tq = p.tq;
    if (t < 0 || m >= min(tq, w.q_len - t * tq) * n_rep)
        return;
    // one pass over the parts in part order; a running largest base
    // rescales what is summed so far
    float mm = -INFINITY, l_sum = 0.f, v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        v[k] = 0.f;
    for (int i0 = 0; i0 < np; i0 += 4) {
        if (i0 > 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const size_t tile = tile0 + 2 * (size_t)(i0 + j < np ? i0 + j : i0);
                ml[j] = __ldcg(&p.ws_ml[tile * C::kRows + m]);
                a[j] = __ldcg(
                    reinterpret_cast<const uint4 *>(p.ws_o + (tile * C::kRows + m) * D + c));
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (i0 + j >= np || !(ml[j].y > 0.f))
                continue;
            if (ml[j].x > mm) {
                const float r = ex2_fast(mm - ml[j].x);        // 0 while mm is -inf
                l_sum *= r;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[k] *= r;
                mm = ml[j].x;
            }
            const float wl = ex2_fast(ml[j].x - mm) * ml[j].y;
            l_sum += wl;
            const uint32_t pa[4] = {a[j].x, a[j].y, a[j].z, a[j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f =
                    __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pa[k]));
                v[2 * k] += wl * f.x;
                v[2 * k + 1] += wl * f.y;
            }
        }
    }
    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
    const int tok = m / n_rep, hh = m - tok * n_rep;
    __nv_bfloat16 *orow =
        p.out + ((size_t)(w.q0 + t * tq + tok) * p.Hq + (size_t)w.g * n_rep + hh) * D + c;
    *reinterpret_cast<uint4 *>(orow) =
        make_uint4(pack_bf16x2(v[0] * inv, v[1] * inv), pack_bf16x2(v[2] * inv, v[3] * inv),
                   pack_bf16x2(v[4] * inv, v[5] * inv), pack_bf16x2(v[6] * inv, v[7] * inv));
}

template <int D>
cudaError_t launch_prefill_d(const PrefillParams &p, int sms, cudaStream_t stream)
{
    using C = PrefillCfg<D>;
    static DeviceOnce attrs;
    const cudaError_t attr_err = attrs.run([] {
        cudaError_t e = cudaFuncSetAttribute(
            prefill_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_kernel<D, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        return e;
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    // one persistent block per SM (each holds all of an SM's tensor memory)
    const int grid = p.n_units < sms ? p.n_units : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = p.split > 1 ? cudaLaunchKernelEx(&cfg, prefill_kernel<D, true>, p)
                                : cudaLaunchKernelEx(&cfg, prefill_kernel<D, false>, p);
    if (e == cudaSuccess && p.split > 1) {
        // the split units' merge, once the kernel above has finished
        cfg.gridDim = dim3((unsigned)(2 * ((p.n_units - p.split_base) / p.split) * (D / 8)));
        cfg.blockDim = dim3(C::kRows);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, prefill_merge_kernel<D>, p);
    }
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library links the runtime only); nullptr when the driver has none.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// A bf16 tensor [rows, mid, D] as the 3-D tiled tensor {D, mid, rows} with
// a box of {64, box_mid, box_rows}, 128-byte swizzled.
bool encode_map(CUtensorMap *map, const void *base, int D, int mid, long long rows, int box_mid,
                int box_rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (fn == nullptr || (reinterpret_cast<uintptr_t>(base) & 15u) != 0)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)mid, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)mid * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_mid, (cuuint32_t)box_rows};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

} // namespace

// Chunks of at most this many pairs of query tiles get a grouped unit list.
constexpr int kGroupMaxPairs = 4;

bool prefill_plan(int B, int Hkv, int tq, int max_q_len, int sms, int D, size_t ws_bytes,
                  PrefillPlan *pl)
{
    *pl = PrefillPlan{};
    pl->split = 1;
    if (B <= 0 || Hkv <= 0 || tq <= 0 || max_q_len <= 0 || sms <= 0)
        return true;                                   // no units
    // the units: pairs of query tiles (max_q_len bounds a chunk's tiles) x
    // rows x kv heads
    const long long tiles = ((long long)max_q_len + tq - 1) / tq;
    const long long pairs = (tiles + 1) / 2;
    const long long units = pairs * B * Hkv;
    if (units > 0x7fffffffLL)
        return false;
    pl->pairs = (int)pairs;
    pl->units = (int)units;
    pl->entries = (int)units;
    pl->split_base = (int)units;
    // rows per group of the unit list.  A chunk of many pairs (a long causal
    // prefill) has units from one to hundreds of key blocks: one group,
    // pair-major, keeps each round's units of about one size.  A chunk of a
    // few pairs (an extend, a short prompt) has units of about one size
    // anyway: groups of about one round of units (SMs / pairs rows) keep the
    // rows in flight few enough to share L2.
    const long long row_heads = (long long)B * Hkv;
    long long grp = row_heads;
    if (pairs <= kGroupMaxPairs) {
        grp = (long long)sms / pairs;
        grp = grp < 1 ? 1 : (grp > row_heads ? row_heads : grp);
    }
    pl->group_rows = (int)grp;
    // the key split: a last round of at most half the SMs (every unit, when
    // they are that few) becomes up to SMs / last entries per unit, as many
    // as the workspace has slots for; every entry of that round leaves its
    // result in its slot and the merge kernel writes the outputs.  A
    // pair-major list of many rounds ends on its smallest pairs (the first
    // query tiles of long chunks: a few key blocks each), so only a grouped
    // list (chunks of a few tile pairs, units of about one size) or a list of
    // one round is cut.
    const long long g0 = units < sms ? units : sms;
    const long long last = units - (units - 1) / g0 * g0;
    const long long slots = (long long)(ws_bytes / prefill_slot_bytes(D));
    long long split = sms / last;
    split = split < kPrefillMaxParts ? split : kPrefillMaxParts;
    split = split < slots / last ? split : slots / last;
    const bool big_last = pairs <= kGroupMaxPairs || units <= g0;
    if (big_last && 2 * last <= sms && split >= 2) {
        pl->split = (int)split;
        pl->split_base = (int)(units - last);
        pl->entries = (int)(units - last + last * split);
    }
    pl->grid = pl->entries < sms ? pl->entries : sms;
    return true;
}

cudaError_t launch_prefill(const PrefillParams &p_in, int D, int max_q_len, void *workspace,
                           size_t ws_bytes, cudaStream_t stream)
{
    // K/V pages by TMA when a page is a power of two >= 8 rows (whole 8-row
    // swizzle atoms; a 128-key block is whole pages or a part of one) and
    // every row index fits the copy's 32-bit coordinate
    PrefillParams p = p_in;
    p.out_align32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
    p.use_tma = 0;
    p.tma_rows = 0;
    const long long rows = (long long)p.num_pages * p.page_size;
    if ((D == 64 || D == 128) && p.ps_shift >= 3 && rows > 0 && rows < (1LL << 31)) {
        const int box_rows = p.page_size < 128 ? p.page_size : 128;
        if (encode_map(&p.tmap_k, p.k_pool, D, p.Hkv, rows, 1, box_rows) &&
            encode_map(&p.tmap_v, p.v_pool, D, p.Hkv, rows, 1, box_rows)) {
            p.use_tma = 1;
            p.tma_rows = box_rows;
        }
    }
    // a query tile (tq tokens x n_rep heads of one kv head) as one box
    p.q_tma = 0;
    if ((D == 64 || D == 128) && p.total_q > 0 && p.n_rep <= 256 && p.tq >= 1 && p.tq <= 256 &&
        encode_map(&p.tmap_q, p.q, D, p.Hq, p.total_q, p.n_rep, p.tq))
        p.q_tma = 1;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    PrefillPlan pl;
    if (!prefill_plan(p.B, p.Hkv, p.tq, max_q_len, sms, D, workspace != nullptr ? ws_bytes : 0,
                      &pl))
        return cudaErrorInvalidValue;
    if (pl.units == 0)
        return cudaSuccess;
    p.pairs = pl.pairs;
    p.n_units = pl.entries;
    p.group_rows = pl.group_rows;
    p.split = pl.split;
    p.split_base = pl.split_base;
    p.ws_o = nullptr;
    p.ws_ml = nullptr;
    if (pl.split > 1) {
        const size_t entries = (size_t)(pl.entries - pl.split_base);
        p.ws_o = static_cast<__nv_bfloat16 *>(workspace);
        p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                             entries * prefill_slot_o_bytes(D));
    }
    return D == 64 ? launch_prefill_d<64>(p, sms, stream) : launch_prefill_d<128>(p, sms, stream);
}

} // namespace pkv
