// pkv_internal.h -- parameter blocks and launchers shared by the .cu files of
// libpkv (not part of the public ABI; see include/pkv.h for that).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// Largest split count any entry point accepts.
constexpr int kMaxSplits = 65536;

// Shape checks common to every entry point (pkv_api.cu).
pkv_status check_dims(const pkv_dims *d);

// One-time set-up of a kernel's function attributes (the opt-in shared
// memory size, the carveout).  Those attributes belong to the current
// device's context, so a process that launches on several devices sets them
// once on each; host threads may launch concurrently, hence the lock.
constexpr int kMaxDevices = 64;

class DeviceOnce {
public:
    template <typename F>
    cudaError_t run(F &&setup)
    {
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 0 || dev >= kMaxDevices)
            return cudaErrorInvalidDevice;
        if (done_[dev].load(std::memory_order_acquire))
            return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev].load(std::memory_order_relaxed))
            return cudaSuccess;
        e = setup();
        if (e == cudaSuccess)
            done_[dev].store(true, std::memory_order_release);
        return e;
    }

private:
    std::mutex mu_;
    std::atomic<bool> done_[kMaxDevices]{};
};

struct AppendParams {
    __nv_bfloat16 *q;
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    __nv_bfloat16 *k_pool;
    __nv_bfloat16 *v_pool;
    const int32_t *kv_indices;
    const int32_t *kv_indptr;
    const int32_t *seq_lens;
    const float *rope;     // [rope_max_pos, D/2, 2] or nullptr
    uint32_t *status;      // nullable
    int B, Hq, Hkv, D, page_size, num_pages, num_indices, max_seq_len;
    int rope_max_pos, rope_q;
    const int32_t *qo_indptr;  // extend: [B+1] chunk offsets (append: unused)
    int total_q;               // extend: tokens in all chunks
};

struct DecodeParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_pool;
    const __nv_bfloat16 *v_pool;
    const int32_t *kv_indices;
    const int32_t *kv_indptr;
    const int32_t *seq_lens;
    float *o_part;         // [B, Hq, S, D]
    float *ml_part;        // [B, Hq, S, 2]
    __nv_bfloat16 *out;    // [B, Hq, D], used when direct != 0
    uint32_t *status;
    int B, Hq, Hkv, n_rep, page_size, ps_shift, num_pages, num_indices;
    int max_seq_len, num_splits, chunk, direct;
    float scale_log2;      // scale * log2(e)
};

// Device-side metadata advance (pkv_advance.cu).
struct AdvanceParams {
    int32_t *seq_lens;
    const int32_t *kv_indptr;
    int32_t *kv_indices;
    const int32_t *free_pages;
    int32_t *free_head;
    uint32_t *status;      // nullable
    int B, page_size, max_seq_len, num_indices, num_free;
};

// Paged ragged prefill / extend (pkv_prefill.cu).
struct PrefillParams {
    const __nv_bfloat16 *q;        // [total_q, Hq, D]
    const int32_t *qo_indptr;      // [B+1]
    const __nv_bfloat16 *k_pool;
    const __nv_bfloat16 *v_pool;
    const int32_t *kv_indices;
    const int32_t *kv_indptr;
    const int32_t *seq_lens;
    __nv_bfloat16 *out;            // [total_q, Hq, D]
    uint32_t *status;              // nullable
    int B, Hq, Hkv, n_rep, page_size, ps_shift, num_pages, num_indices, max_seq_len, total_q;
    int tq;                        // query tokens per block: 128 / n_rep
    float scale_log2;
    // the pools as 3-D tiled tensors {D, Hkv, pages x page_size} with a box of
    // {64, 1, tma_rows} and 128-byte swizzle (use_tma != 0; set by
    // launch_prefill when the page size is a power of two >= 8)
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    int use_tma;
    int tma_rows;                  // min(page_size, 128)
    // q as {D, Hq, total_q} with a box of {64, n_rep, tq}: one query tile's
    // rows (token-major, head-minor), 128-byte swizzled (q_tma != 0)
    CUtensorMap tmap_q;
    int q_tma;
    // the units of work (set by launch_prefill): pairs of query tiles per
    // chunk (from max_q_len) and pairs x B x Hkv
    int pairs;
    int n_units;                   // entries of the list: units, then split parts
    int group_rows;                // rows per group of the unit list
    // the key split (split > 1): entries [split_base, n_units) are the parts
    // of the list's last units, split to a unit; entry e's tile x leaves its
    // normalised rows at ws_o [(2 e + x) x 128 + row][D] and each row's
    // (base, l) at ws_ml [(2 e + x) x 128 + row] for the merge kernel
    int split;
    int split_base;
    __nv_bfloat16 *ws_o;
    float2 *ws_ml;
    // out is 32-byte aligned: rows are stored with 32-byte stores (set by
    // launch_prefill; otherwise 16-byte stores, each lane its own row)
    int out_align32;
};

// The prefill's key split.  When the unit list's last round would leave at
// least half the SMs idle, its units are cut along their key blocks into
// parts on separate SMs (at most kPrefillMaxParts, each of at least
// kPrefillMinPartBlocks blocks).
constexpr int kPrefillMaxParts = 16;
constexpr int kPrefillMinPartBlocks = 2;
// Workspace: per entry of the split round, two tiles of 128 bf16 rows of D
// (all entries' rows first) and two tiles of 128 fp32 (base, l) pairs; for
// up to kPrefillMaxSms SMs.
constexpr int kPrefillMaxSms = 1024;
inline size_t prefill_slot_o_bytes(int D) { return (size_t)2 * 128 * D * 2; }
inline size_t prefill_slot_bytes(int D) { return prefill_slot_o_bytes(D) + (size_t)2 * 128 * 8; }

// Persistent token-balanced decode (pkv_fused.cu).
constexpr int kFusedMaxRows = 4096;     // virtual rows whose prefix sums fit in smem
constexpr int kFusedMinTokens = 64;     // fewest tokens a block is given
// Partition weight of a row beyond its tokens: a block pays a fixed cost at
// each row it starts (page-table window, q block, partial write), measured
// at about 1.8 us per extra row, the time of ~20 streamed tokens.  Charging
// it in the partition gives blocks that cross more row boundaries fewer
// tokens; 32 measured best of {0, 16, 32, 48} on the serving mixes.
constexpr int kFusedRowCost = 32;

struct FusedParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_pool;
    const __nv_bfloat16 *v_pool;
    const int32_t *kv_indices;
    const int32_t *kv_indptr;
    const int32_t *seq_lens;
    __nv_bfloat16 *out;
    float *o_part;         // [(grid + Bv) * HQV, D]  piece partials
    float *ml_part;        // [(grid + Bv) * HQV, 2]
    int32_t *row_info;     // [Bv, 2]: first block, piece count
    uint32_t *status;
    int B, Hq, Hkv, n_rep, page_size, ps_shift, num_pages, num_indices, max_seq_len;
    int Bv;                // virtual rows: (Hkv / hpc) head groups x B
    int row_cost;          // partition weight of a non-empty row beyond its tokens
    int hpc;               // kv heads per block (1, 2, 4 or 8)
    float scale_log2;
    // fused step: the new token (k_new, v_new at position seq_len - 1) is
    // rotated, written to its pool slot and attended from shared memory; q
    // is rotated in registers.  step == 0: plain decode over the pool.
    int step;
    __nv_bfloat16 *k_pool_w;          // the pools, writable (step only)
    __nv_bfloat16 *v_pool_w;
    const __nv_bfloat16 *k_new;       // [B, Hkv, D]
    const __nv_bfloat16 *v_new;
    const float *rope;                // [rope_max_pos, D/2, 2] or nullptr
    int rope_max_pos;
    // limit of the waits that hand a stage or the q block between the
    // producer and the consumers (normally the full ~2 s; shortened only by
    // the testing call).  Waits for copies already issued keep the full limit.
    unsigned long long handoff_wait_ns;
    // the step's plan (paged_decode_plan) or nullptr: the partition computed
    // at the kernel's start instead
    const int32_t *plan;
    // unplanned calls: where to leave the partition as the step's plan
    // (nullptr: nowhere)
    int32_t *plan_out;
};

// Threads of a plan block.
constexpr int kPlanThreads = 256;
// int32 words of the plan for Bv virtual rows and a grid of `grid` blocks.
inline size_t plan_words(int Bv, int grid)
{
    return 16 + (((size_t)Bv + 1 + 3) & ~(size_t)3) + (size_t)72 * grid;
}

// The hand-off wait limit launches use (pkv_testing_set_handoff_wait_ns).
unsigned long long handoff_wait_ns();

struct PieceCombineParams {
    const float *o_part;
    const float *ml_part;
    const int32_t *row_info;
    __nv_bfloat16 *out;
    int B, Bv, Hq, HQV;
    int planned;           // row_info written by the plan kernel (read before the wait)
    // paged_decode_step_advance: one extra block runs the metadata advance
    // (adv.seq_lens == nullptr: none)
    AdvanceParams adv;
};

struct CombineParams {
    const float *o_part;
    const float *ml_part;
    __nv_bfloat16 *out;
    int B, Hq, D, num_splits;
};

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream);
cudaError_t launch_extend(const AppendParams &p, cudaStream_t stream);
cudaError_t launch_advance(const AdvanceParams &p, cudaStream_t stream);
// one persistent block per SM over the units (pairs of query tiles x B x Hkv)
// The prefill's list for a launch (host only): units of tile pairs, their
// grouping, and the key split of the last round.
struct PrefillPlan {
    int pairs;       // tile pairs a chunk of max_q_len has
    int units;       // pairs x B x Hkv (0: nothing to run)
    int group_rows;  // rows per group of the list
    int entries;     // units, or with a split units - last + last x split
    int split;       // parts per unit of the last round (1: no split)
    int split_base;  // the last round's first entry
    int grid;        // blocks: min(entries, sms)
};
// false when the list would exceed 2^31 - 1 units.  ws_bytes: the key
// split's workspace (0: none).
bool prefill_plan(int B, int Hkv, int tq, int max_q_len, int sms, int D, size_t ws_bytes,
                  PrefillPlan *pl);

// workspace (nullable, 256-byte aligned, ws_bytes long) enables the key
// split with as many part slots as it holds.
cudaError_t launch_prefill(const PrefillParams &p, int D, int max_q_len, void *workspace,
                           size_t ws_bytes, cudaStream_t stream);
// table[0..B] = 0..B (kv_indptr), table[B+1+b] = idx ? idx[b] : b (kv_indices)
cudaError_t launch_contig_table(const int32_t *idx, int B, int32_t *table, cudaStream_t stream);
cudaError_t launch_rope_table(float *cos_sin, int max_pos, int D, double base,
                              cudaStream_t stream);
cudaError_t launch_split_decode(const DecodeParams &p, int D, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);
cudaError_t launch_fused_decode(const FusedParams &p, int D, int grid, cudaStream_t stream);
cudaError_t launch_piece_combine(const PieceCombineParams &p, int D, int grid_blocks,
                                 cudaStream_t stream);
// The per-step plan for the decode kernel's grid of `grid` blocks; p carries
// the shape, the tables, row_info and the status word.
cudaError_t launch_decode_plan(const FusedParams &p, int grid, int32_t *plan,
                               cudaStream_t stream);
int fused_heads_per_block(int Hkv);

// Resident split-decode blocks per SM for head dim D (shared-memory bound).
int split_decode_blocks_per_sm(int D);

} // namespace pkv
