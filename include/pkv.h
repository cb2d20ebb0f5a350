/*
 * pkv.h -- C ABI of libpkv: paged GQA decode attention for one NVIDIA GB300
 * (sm_103a).
 *
 * The operation (AstrAI commit log, page "compare v1.3.12..6f09b1d",
 * astrai/extension/attention_ops.py, docstring of attn_paged_decode, and
 * astrai/extension/attention_backend.py, CudaBackend.fwd_decode): each of B
 * query rows holds one new token.  The token's K/V are written into its slot
 * of a paged pool; then each of its Hq query heads attends, with
 * softmax(q K^T * scale) V, over all seq_lens[b] tokens of its row, reading
 * kv head h / (Hq/Hkv) (grouped-query attention, repeat_kv on the same page).
 * The attention is computed split-KV: each split of a row writes a partial
 * (normalised output, max, sum) and a combine pass merges them (commits by
 * author: "single combine kernel", "split partials", "compute_num_splits").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    allocates nothing, holds no per-call state, never synchronises and never
 *    prints.  Kernels are launched asynchronously on `stream` (NULL = the
 *    legacy default stream), so every call can be captured in a CUDA graph.
 *  - bf16 means IEEE bfloat16; every bf16 array must be 16-byte aligned and
 *    densely packed in the layout given.  Tables are int32.
 *  - Layouts:
 *      q, out          [B, Hq, D]                  bf16
 *      k_new, v_new    [B, Hkv, D]                 bf16
 *      k_pool, v_pool  [num_pages, page_size, Hkv, D] bf16
 *      seq_lens        [B]    tokens of row b INCLUDING this step's new token
 *      kv_indptr       [B+1]  row b's pages are kv_indices[kv_indptr[b] ..
 *                             kv_indptr[b+1]), in logical order; it needs at
 *                             least ceil(seq_lens[b] / page_size) of them
 *      kv_indices      [num_indices] physical page ids in [0, num_pages)
 *    Logical token t of row b lives in page kv_indices[kv_indptr[b] +
 *    t / page_size], slot t % page_size (compare v1.3.12..6f09b1d,
 *    astrai/inference/core/cache.py, PagePool._extend_slot).
 *  - Host-side checks return a pkv_status before anything is launched.
 *    Device-side checks never trap: a bad table entry or length is skipped
 *    (reading page 0 instead, so nothing outside the pool is touched) and
 *    recorded by OR-ing a PKV_FLAG_* bit into the 32-bit status word at
 *    offset 0 of the workspace.  The word is sticky: clear it with
 *    pkv_workspace_init and read it back with a device-to-host copy.
 *  - Launch failures come back as PKV_ERR_LAUNCH (cudaGetLastError).
 *  - Supported shapes: D in {64, 128}; Hq % Hkv == 0; 1 <= Hq/Hkv <= 16;
 *    page_size >= 1 (powers of two take a shift, others a division);
 *    1 <= B <= 65535; Hkv <= 65535.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,        /* null/misaligned pointer, bad shape  */
    PKV_ERR_UNSUPPORTED = -2,        /* valid but not built (e.g. D = 96)   */
    PKV_ERR_WORKSPACE_TOO_SMALL = -3,
    PKV_ERR_LAUNCH = -4              /* a CUDA launch reported an error     */
} pkv_status;

/* Device status word bits (workspace offset 0). */
#define PKV_FLAG_BAD_PAGE 0x1u  /* page id outside [0,num_pages), kv_indptr
                                   outside [0,num_indices], or a row whose
                                   table is shorter than its length         */
#define PKV_FLAG_BAD_LEN  0x2u  /* seq_lens[b] < 0 or > max_seq_len         */
#define PKV_FLAG_BAD_POS  0x4u  /* new-token position >= RoPE table rows    */
#define PKV_FLAG_TIMEOUT  0x8u  /* an internal copy wait gave up (~2 s)     */
#define PKV_FLAG_NO_PAGE  0x10u /* paged_kv_advance: free list empty, or the
                                   row's page-table capacity is full        */

typedef struct {
    int B;            /* query rows in the batch                           */
    int Hq;           /* query heads                                        */
    int Hkv;          /* kv heads; query head h reads kv head h/(Hq/Hkv)    */
    int D;            /* head dim, 64 or 128                                */
    int page_size;    /* tokens per page                                    */
    int num_pages;    /* pages in each pool (>= 1)                          */
    int num_indices;  /* length of kv_indices                               */
    int max_seq_len;  /* upper bound on every seq_lens[b]; with num_splits
                         it fixes the split grid, so a captured graph stays
                         valid while lengths change below it                */
    float scale;      /* softmax scale; normally 1/sqrt(D)                  */
} pkv_dims;

/* ---- planning (host only, no CUDA calls) -------------------------------- */

/* num_splits, two readings.  paged_decode_attn / paged_decode_step on the
 * persistent path (at most 4096 rows x kv-head groups, the usual case): the
 * number of persistent blocks; all rows' tokens laid end to end are cut into
 * num_splits equal ranges (never below 64 tokens each), so a row is split
 * into as many pieces as ranges it touches -- a single row into up to
 * num_splits.  paged_decode_partials, and paged_decode_attn on other shapes:
 * the per-row split count, each split covering `chunk` tokens (below). */

/* Tokens per split of the per-row layout:
 * ceil(ceil(max_seq_len / num_splits) / 16) * 16.  Split s of row b covers
 * logical tokens [s*chunk, min((s+1)*chunk, seq_lens[b])).  Returns 0 for
 * invalid arguments. */
int pkv_split_chunk(const pkv_dims *dims, int num_splits);

/* Workspace bytes for num_splits: a 256-byte header (status word first),
 * per-row bookkeeping, the per-step plan (paged_decode_plan), a [B, Hq, D]
 * bf16 scratch, and room for either
 * partial layout (the per-row one [B, Hq, S, 2] + [B, Hq, S, D] fp32, or the
 * persistent path's pieces), each region 256-byte aligned.  Returns 0 for
 * invalid arguments. */
size_t pkv_workspace_bytes(const pkv_dims *dims, int num_splits);

/* Byte offsets of the per-row layout's ml_part and o_part (as written by
 * paged_decode_partials) inside the workspace. */
pkv_status pkv_workspace_layout(const pkv_dims *dims, int num_splits,
                                size_t *ml_offset, size_t *o_offset);

/* Split count for this shape on a GPU with num_sms SMs.  Persistent path:
 * one block per SM, fewer when max_seq_len x rows gives under 64 tokens a
 * block.  Per-row path: enough (split, kv head, row) blocks for a few waves,
 * never splitting below 256 tokens (commits by author, "compute_num_splits
 * ... undersplitting at large batch"; "bandwidth saturates near 256-512
 * total blocks").  Writes the count and the workspace size it needs. */
pkv_status pkv_plan(const pkv_dims *dims, int num_sms, int *num_splits,
                    size_t *ws_bytes);

/* ---- set-up -------------------------------------------------------------- */

/* Zero the workspace status word (stream-ordered memset; no allocation). */
pkv_status pkv_workspace_init(void *workspace, size_t ws_bytes, pkv_stream_t stream);

/* Fill the RoPE table cos_sin [max_pos, D/2, 2] fp32 with (cos, sin) of
 * pos * base^(-2i/D), computed in double and rounded once to fp32 (commits
 * by author: "cos/sin freqs_cis table"). */
pkv_status pkv_rope_table(float *cos_sin, int max_pos, int D, double base,
                          pkv_stream_t stream);

/* ---- the hot path --------------------------------------------------------- */

/* (1) Fused RoPE + K/V append.  For each row with L = seq_lens[b] > 0, the
 * new token's position is p = L-1 (compare v1.3.12..6f09b1d,
 * astrai/inference/core/task.py next_pos, and cache.py bind_tasks writing at
 * seq_len - 1).  Each K head vector of k_new[b] is rotated by p on
 * interleaved pairs (x[2i], x[2i+1]) -> (x[2i] c - x[2i+1] s,
 * x[2i] s + x[2i+1] c), (c, s) = rope_cos_sin[p][i], in fp32, rounded to
 * bf16 and stored at the token's slot; V is stored unchanged.  With rope_q,
 * every query head of row b is rotated the same way, in place.
 * rope_cos_sin == NULL skips rotation.  Rows with L = 0 are skipped.
 * status (nullable) receives PKV_FLAG_* bits; an offending row writes
 * nothing. */
pkv_status paged_kv_append(const pkv_dims *dims, void *q, const void *k_new,
                           const void *v_new, void *k_pool, void *v_pool,
                           const int32_t *kv_indices, const int32_t *kv_indptr,
                           const int32_t *seq_lens, const float *rope_cos_sin,
                           int rope_max_pos, int rope_q, uint32_t *status,
                           pkv_stream_t stream);

/* (2)+(3) Split-KV decode attention.  out[b, h] = softmax(q[b,h] K^T * scale)
 * V over the row's seq_lens[b] tokens (all of them: decode is causal and the
 * query is the last token).  Rows with seq_lens[b] = 0 give zeros.
 * Persistent path: one token-balanced kernel (a piece that is a whole row
 * writes out directly) plus, when num_splits > 1, the piece combine.  Other
 * shapes: the per-(split, kv head, row) kernel, plus decode_combine when
 * num_splits > 1.  workspace must be 256-byte aligned and hold
 * pkv_workspace_bytes(dims, num_splits) bytes; its status word must have
 * been zeroed once (pkv_workspace_init). */
pkv_status paged_decode_attn(const pkv_dims *dims, const void *q,
                             const void *k_pool, const void *v_pool,
                             const int32_t *kv_indices, const int32_t *kv_indptr,
                             const int32_t *seq_lens, int num_splits,
                             void *workspace, size_t ws_bytes, void *out,
                             pkv_stream_t stream);

/* (1)+(2)+(3) in one pass: the whole decode step.  Appends each row's new
 * token exactly as paged_kv_append does (K rotated by position seq_len - 1
 * and rounded to bf16, V copied, both into the token's slot of the pools)
 * and computes out exactly as paged_decode_attn does, with q rotated by the
 * same position.  q itself is NOT modified (its rotation stays internal).
 * For shapes the persistent kernel serves (at most 4096 rows x kv-head
 * groups) it is one launch plus the combine: the new token is rotated in
 * the decode kernel and attended from shared memory, and q is rotated in
 * registers.  Otherwise it runs a rotated copy of q (in the workspace), the
 * append and the split decode.  rope_cos_sin == NULL: no rotation.
 * Device-side errors set the PKV_FLAG_* bits of the workspace status word. */
pkv_status paged_decode_step(const pkv_dims *dims, const void *q, const void *k_new,
                             const void *v_new, void *k_pool, void *v_pool,
                             const int32_t *kv_indices, const int32_t *kv_indptr,
                             const int32_t *seq_lens, const float *rope_cos_sin,
                             int rope_max_pos, int num_splits, void *workspace,
                             size_t ws_bytes, void *out, pkv_stream_t stream);

/* ---- the per-step plan --------------------------------------------------- */

/* The decode metadata built once per step and reused by every layer's call
 * of that step (commits by author: kv_indptr built once per step instead of
 * per layer; the per-step metadata precompute of the decode path).  Writes
 * into the workspace the partition that paged_decode_attn and
 * paged_decode_step compute at the start of each call on the persistent
 * path: the rows' prefix sums, each row's first block and piece count, and
 * for each of the num_splits blocks its first row and that row's 64-entry
 * page-table window.  A call of paged_decode_attn_planned or
 * paged_decode_step_planned with the same dims and num_splits on this
 * workspace then starts streaming after one round trip to memory instead of
 * three, and its piece combine reads the row ranges while the decode grid
 * finishes.  One launch of num_splits blocks; graph-capturable; allocates
 * nothing.  The plan stays valid until seq_lens, kv_indptr, kv_indices, dims
 * or num_splits change: the caller plans again after any of them changes
 * (once per decode step).  paged_decode_attn and paged_decode_step on the
 * persistent path leave the partition they compute in the workspace as the
 * same plan, so a step whose first layer calls them needs no separate
 * paged_decode_plan before its later layers' planned calls.  A planned call on a plan made for another grid or
 * shape falls back to computing the partition itself; on a plan made for
 * other lengths or tables it reads no memory out of bounds but its output is
 * undefined.  Length and table checks run in the plan and set PKV_FLAG_*
 * bits of the workspace status word.  Shapes off the persistent path need
 * no plan: the call returns PKV_OK and writes nothing.  Arguments as in
 * paged_decode_attn. */
pkv_status paged_decode_plan(const pkv_dims *dims, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *seq_lens,
                             int num_splits, void *workspace, size_t ws_bytes,
                             pkv_stream_t stream);

/* paged_decode_attn on the workspace's plan (paged_decode_plan).  Arguments
 * and results are those of paged_decode_attn, bit for bit. */
pkv_status paged_decode_attn_planned(const pkv_dims *dims, const void *q,
                                     const void *k_pool, const void *v_pool,
                                     const int32_t *kv_indices, const int32_t *kv_indptr,
                                     const int32_t *seq_lens, int num_splits,
                                     void *workspace, size_t ws_bytes, void *out,
                                     pkv_stream_t stream);

/* paged_decode_step on the workspace's plan (paged_decode_plan).  Arguments
 * and results are those of paged_decode_step, bit for bit; the step's new
 * token does not change the plan (its length is already counted). */
pkv_status paged_decode_step_planned(const pkv_dims *dims, const void *q, const void *k_new,
                                     const void *v_new, void *k_pool, void *v_pool,
                                     const int32_t *kv_indices, const int32_t *kv_indptr,
                                     const int32_t *seq_lens, const float *rope_cos_sin,
                                     int rope_max_pos, int num_splits, void *workspace,
                                     size_t ws_bytes, void *out, pkv_stream_t stream);

/* The split kernel alone: always writes the partials (never out), for any
 * num_splits >= 1.  Partial (b, h, s): o_part = the split's softmax-weighted
 * V average (normalised), ml_part = (m, l) with m = max of scale * q.k over
 * the split (natural-log units) and l = sum exp(scale * q.k - m); an empty
 * split writes (m, l) = (-inf, 0) and leaves o_part unwritten. */
pkv_status paged_decode_partials(const pkv_dims *dims, const void *q,
                                 const void *k_pool, const void *v_pool,
                                 const int32_t *kv_indices,
                                 const int32_t *kv_indptr,
                                 const int32_t *seq_lens, int num_splits,
                                 void *workspace, size_t ws_bytes,
                                 pkv_stream_t stream);

/* (3) Combine: for each (b, h), M = max m_s over splits with l_s > 0,
 * w_s = l_s exp(m_s - M), out = sum w_s o_s / sum w_s, rounded to bf16;
 * all-empty -> 0.  o_part [B, Hq, S, D], ml_part [B, Hq, S, 2] fp32, as
 * written by the split kernel (or by any producer of the same layout). */
pkv_status decode_combine(const pkv_dims *dims, const float *o_part,
                          const float *ml_part, int num_splits, void *out,
                          pkv_stream_t stream);

/* ---- prefill / extend ----------------------------------------------------- */

/* Paged ragged prefill / extend attention (compare v1.3.12..6f09b1d,
 * astrai/extension/attention_ops.py, attn_paged_prefill: "SGLang-style paged
 * prefill (ragged batch ...)"; attn_prefill's causal offset kv_len - q_len).
 * q [total_q, Hq, D] bf16 holds every row's query chunk back to back;
 * qo_indptr [B+1] int32 is the prefix sum of the chunk lengths (0 ..
 * total_q).  Row b's chunk is the last q_len = qo_indptr[b+1] - qo_indptr[b]
 * of its L = seq_lens[b] tokens, whose K/V must already be in the pools
 * (same page table as the decode calls), so query i sits at position
 * L - q_len + i and attends keys 0 .. that position:
 *   out[qo_indptr[b] + i, h] = softmax(scale q K^T) V over those keys, kv
 *   head h / (Hq/Hkv), fp32 softmax, bf16 output [total_q, Hq, D].
 * dims->scale must be > 0.
 * max_q_len (host int, >= every chunk length; the pages' "max per-request
 * q_len ... for grid computation") sizes the grid.  A row with q_len < 0 or
 * > L, L > max_seq_len, or a chunk longer than max_q_len sets
 * PKV_FLAG_BAD_LEN and its outputs are left unwritten; bad page ids set
 * PKV_FLAG_BAD_PAGE (page 0 is read instead).  B * Hkv <= 65535 (else
 * PKV_ERR_UNSUPPORTED).  status (device, nullable) receives the flags.  No
 * workspace; graph-capturable.  Runs on the 5th-generation tensor cores
 * (tcgen05.mma, accumulators in tensor memory); at D = 128 each block holds
 * all 512 tensor-memory columns of its SM while it runs, so kernels of other
 * streams that allocate tensor memory wait for it on that SM. */
pkv_status paged_prefill_attn(const pkv_dims *dims, const void *q, const int32_t *qo_indptr,
                              int total_q, int max_q_len, const void *k_pool, const void *v_pool,
                              const int32_t *kv_indices, const int32_t *kv_indptr,
                              const int32_t *seq_lens, void *out, uint32_t *status,
                              pkv_stream_t stream);

/* paged_prefill_attn with a workspace, which lets it split keys: the pages'
 * split-KV (partials over ranges of keys merged by their (max, sum), as
 * decode_combine merges decode splits), applied to prefill's units of work.
 * Those units are pairs of query tiles of one (row, kv head); one block per
 * SM takes one unit per round.  When the last round would fill at most half
 * the SMs (every unit, when they are that few), each of its units runs as
 * up to min(16, SMs / units in that round, n / 2) parts over consecutive
 * ranges of its n key blocks, each on an SM of its own.  Every entry of that
 * round leaves its rows in a workspace slot, normalised on a base of its own
 * and rounded to bf16 as outputs are, with each row's fp32 (base, l); a
 * second, small kernel merges each unit's parts in part order and writes
 * its outputs.  The result differs from paged_prefill_attn's by that one
 * extra bf16 rounding of each part (within one bf16 step), and is the same
 * bits from call to call.
 * workspace: device scratch, 256-byte aligned, ws_bytes long, needing no
 * initialisation; pkv_prefill_workspace_bytes(D, SMs) has a slot for every
 * entry a round can hold.  A smaller workspace gets fewer parts; NULL, or
 * one with fewer slots than two per unit of that round, runs
 * paged_prefill_attn.  Calls that share a workspace must not overlap on the
 * GPU.  Other arguments, errors and flags are paged_prefill_attn's;
 * graph-capturable (one or two kernel launches). */
pkv_status paged_prefill_attn_ws(const pkv_dims *dims, const void *q, const int32_t *qo_indptr,
                                 int total_q, int max_q_len, const void *k_pool,
                                 const void *v_pool, const int32_t *kv_indices,
                                 const int32_t *kv_indptr, const int32_t *seq_lens,
                                 void *workspace, size_t ws_bytes, void *out, uint32_t *status,
                                 pkv_stream_t stream);

/* Bytes of the paged_prefill_attn_ws workspace with a slot for each of
 * num_sms SMs (the most entries a round holds) at head dim D: per slot two
 * tiles of 128 bf16 rows of D and 128 fp32 (base, l) pairs,
 * num_sms x (512 D + 2048) bytes (9.8 MiB at D = 128 on 152 SMs).  0 for D
 * other than 64 or 128, or num_sms outside 1..1024. */
size_t pkv_prefill_workspace_bytes(int D, int num_sms);

/* The list of work paged_prefill_attn / paged_prefill_attn_ws would launch
 * on num_sms SMs (host only; no device is touched), for planning and tests.
 * plan (host, 7 int32) receives:
 *   [0] pairs      tile pairs in a chunk of max_q_len (a tile is 128 / n_rep
 *                  tokens x n_rep query heads)
 *   [1] units      pairs x B x Hkv
 *   [2] group_rows rows (b, kv head) per group of the list: all of them
 *                  (pair-major) when a chunk has more than 4 pairs
 *   [3] entries    units, or with a key split units - last + last x split
 *   [4] split      parts per unit of the last round (1: no split); a split
 *                  needs ws_bytes > 0, a last round of at most num_sms / 2
 *                  units, and a grouped list or a single round
 *   [5] split_base the last round's first entry
 *   [6] grid       blocks launched: min(entries, num_sms)
 * ws_bytes: the workspace paged_prefill_attn_ws would get (0: none).  Errors:
 * check_dims's, PKV_ERR_INVALID_ARG for a null plan, max_q_len < 0 or
 * num_sms outside 1..1024, PKV_ERR_UNSUPPORTED past 2^31 - 1 units. */
pkv_status pkv_prefill_plan(const pkv_dims *dims, int max_q_len, int num_sms, size_t ws_bytes,
                            int32_t *plan);

/* Extend: the K/V write of a prefill / extend chunk, the multi-token form of
 * paged_kv_append (compare v1.3.12..6f09b1d, attention_backend.py: the
 * prefill path stores every new token's K/V at its slot).  Row b's
 * q_len = qo_indptr[b+1] - qo_indptr[b] new tokens are the last q_len of its
 * L = seq_lens[b] (seq_lens already count them): token i of the chunk (input
 * row qo_indptr[b] + i of k_new / v_new [total_q, Hkv, D] and q
 * [total_q, Hq, D]) sits at position L - q_len + i.  K is rotated by that
 * position as paged_kv_append does, V copied, both stored at the token's
 * slot; with rope_q its query heads are rotated in place (q may be NULL
 * otherwise).  A row with q_len < 0 or > L, or L > max_seq_len, sets
 * PKV_FLAG_BAD_LEN and writes nothing; page and position errors as for
 * paged_kv_append.  One block per new token; graph-capturable.  Followed by
 * paged_prefill_attn on the same chunks, it is the whole extend step. */
pkv_status paged_kv_extend(const pkv_dims *dims, void *q, const void *k_new, const void *v_new,
                           const int32_t *qo_indptr, int total_q, void *k_pool, void *v_pool,
                           const int32_t *kv_indices, const int32_t *kv_indptr,
                           const int32_t *seq_lens, const float *rope_cos_sin,
                           int rope_max_pos, int rope_q, uint32_t *status,
                           pkv_stream_t stream);

/* ---- contiguous K/V cache -------------------------------------------------- */

/* Decode (or, with k_new/v_new, the whole decode step) over a contiguous
 * K/V cache, the pages' ContigKV layout (compare v1.3.12..6f09b1d,
 * attention_backend.py: "Read K/V directly from flat pool via
 * cache_batch_idx + cache_seqlens"; commits by author, "add attn_kv_source.cuh
 * with ContigKV/PagedKV addressing policies").
 * k_cache, v_cache: [num_slots, cache_len, Hkv, D] bf16 with
 * dims->num_pages = num_slots and dims->page_size = cache_len.  Row b reads
 * slot cache_batch_idx[b] (NULL: slot b) over its seq_lens[b] tokens, so
 * the cache is a paged pool with one page of cache_len tokens per row.
 * dims->num_indices is ignored.  The call writes that one-entry table into
 * the workspace (a region every workspace has) and runs paged_decode_attn,
 * or paged_decode_step when k_new and v_new are given (then the new token
 * is written at seq_lens[b] - 1 of its slot; rope_cos_sin / rope_max_pos as
 * for that call).  Errors and results are those calls'; a slot id outside
 * [0, num_slots) sets PKV_FLAG_BAD_PAGE. */
pkv_status decode_attn_contig(const pkv_dims *dims, const void *q, const void *k_new,
                              const void *v_new, void *k_cache, void *v_cache,
                              const int32_t *cache_batch_idx, const int32_t *seq_lens,
                              const float *rope_cos_sin, int rope_max_pos, int num_splits,
                              void *workspace, size_t ws_bytes, void *out,
                              pkv_stream_t stream);

/* decode_attn_contig for the later layers of a step: it reuses the one-entry
 * table and the plan (paged_decode_plan) that the step's first
 * decode_attn_contig call left in this workspace, so it launches no table
 * kernel and runs the planned decode (or step).  Valid while dims,
 * num_splits, cache_batch_idx and seq_lens are those of that first call.
 * Arguments and results are those of decode_attn_contig, bit for bit. */
pkv_status decode_attn_contig_planned(const pkv_dims *dims, const void *q, const void *k_new,
                                      const void *v_new, void *k_cache, void *v_cache,
                                      const int32_t *cache_batch_idx, const int32_t *seq_lens,
                                      const float *rope_cos_sin, int rope_max_pos,
                                      int num_splits, void *workspace, size_t ws_bytes,
                                      void *out, pkv_stream_t stream);

/* ---- the decode loop on the device --------------------------------------- */

/* Advance the decode metadata by one token per live row, on the device, so
 * that a loop of decode steps can be one CUDA graph with no host work
 * between steps.  It does what the pages' host code does at each steady-state
 * step (compare v1.3.12..6f09b1d, astrai/inference/core/cache.py:
 * PagePool.task_extend / _extend_slot claim the new token's slot, taking a
 * fresh page from the allocator when the position starts a page, and set the
 * length to pos + 1; bind_tasks' steady-state branch adds one to every
 * row's length in place; commits by author, "DecodeBindCache: bind_tasks
 * increments seq_lens/kv_indptr").
 *
 * For each row b with L = seq_lens[b] > 0 (rows with 0 are idle and left
 * alone), the new token's position is pos = L:
 *   - pos >= max_seq_len: PKV_FLAG_BAD_LEN, row unchanged;
 *   - pos % page_size == 0 (the token starts a page): the row takes the next
 *     free page and kv_indices[kv_indptr[b] + pos / page_size] = that page.
 *     Rows take pages in increasing b from free_pages[*free_head],
 *     free_pages[*free_head + 1], ..., so the assignment is deterministic.
 *     If the row's capacity (kv_indptr[b+1] - kv_indptr[b] entries) has no
 *     entry pos / page_size, or the list has run out (index >= num_free), the
 *     row is unchanged and PKV_FLAG_NO_PAGE is set;
 *   - otherwise seq_lens[b] = pos + 1.
 * *free_head advances by the pages taken.  The page table therefore needs
 * room to grow: a strided layout (kv_indptr[b] = b * cap) does it.
 * kv_indptr is only read.
 *
 * Then paged_decode_step (or paged_kv_append) writes the new token at
 * seq_lens[b] - 1, as usual.  seq_lens, kv_indices and free_head are device
 * int32 arrays the call reads and writes; free_pages (num_free entries, may
 * be NULL when num_free == 0) is read; status (device, nullable) receives
 * PKV_FLAG_* bits.  Page ids are not range-checked here; the decode checks
 * every id it reads.  One launch of one block; graph-capturable. */
pkv_status paged_kv_advance(const pkv_dims *dims, int32_t *seq_lens,
                            const int32_t *kv_indptr, int32_t *kv_indices,
                            const int32_t *free_pages, int num_free, int32_t *free_head,
                            uint32_t *status, pkv_stream_t stream);

/* paged_decode_step followed by paged_kv_advance, for a decode loop: the
 * step attends and appends at the current seq_lens, then the metadata moves
 * on to the next step's token (the same two host steps of the pages as
 * paged_kv_advance, run after the step instead of before it).  Results are
 * bit-identical to the two calls in that order.  Arguments are those of the
 * two calls; the advance's PKV_FLAG_* bits go to the workspace status word.
 * On the persistent path with num_splits > 1 the advance is one extra block
 * of the piece-combine launch (that launch starts after the decode grid has
 * completed, and its other blocks never read the metadata), so the step
 * stays two launches; otherwise it is paged_decode_step plus the one-block
 * advance launch.  A loop starts with one paged_kv_advance and then calls
 * this once per step; the state after K of these calls is that after K + 1
 * advances and K steps.  Graph-capturable. */
pkv_status paged_decode_step_advance(const pkv_dims *dims, const void *q, const void *k_new,
                                     const void *v_new, void *k_pool, void *v_pool,
                                     int32_t *kv_indices, const int32_t *kv_indptr,
                                     int32_t *seq_lens, const float *rope_cos_sin,
                                     int rope_max_pos, int num_splits, void *workspace,
                                     size_t ws_bytes, void *out, const int32_t *free_pages,
                                     int num_free, int32_t *free_head, pkv_stream_t stream);

/* ---- for callers that cannot allocate ------------------------------------ */

/* Size of the library-held scratch used by paged_decode_attn_noalloc. */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

/* paged_decode_attn without a caller workspace.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory
 * (a runtime whose memory pool owns every allocation, a plugin host that
 * forbids allocation while it executes, a path that must not fail on
 * out-of-memory), so they cannot provide the workspace the other calls need.
 * The workspace is a 16 MiB array the library keeps in device memory on
 * every GPU that loads it, until the process exits; this call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Arguments and results are those of paged_decode_attn.  A shape whose
 * workspace (pkv_workspace_bytes(dims, num_splits)) exceeds
 * PKV_NOALLOC_SCRATCH_BYTES is rejected with PKV_ERR_WORKSPACE_TOO_SMALL.
 * status (nullable, device, 4-byte aligned) receives this call's PKV_FLAG_*
 * word; the word is cleared at the start of every call.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array and keep the last call's contents:
 * calls that can overlap on the GPU (other streams, other threads) race and
 * must be serialised by the caller. */
pkv_status paged_decode_attn_noalloc(const pkv_dims *dims, const void *q,
                                     const void *k_pool, const void *v_pool,
                                     const int32_t *kv_indices, const int32_t *kv_indptr,
                                     const int32_t *seq_lens, int num_splits, void *out,
                                     uint32_t *status, pkv_stream_t stream);

/* ---- testing -------------------------------------------------------------- */

/* Test-only: the time limit, in nanoseconds, of the waits that hand a stage
 * or a q block between the decode kernel's copy warp and its compute warps
 * (default and maximum: 2,000,000,000).  A shorter limit makes those waits
 * give up while data is still in flight, so tests can drive the timeout path:
 * the kernel then sets PKV_FLAG_TIMEOUT in the status word, lets every copy
 * it has issued land (those waits keep the full limit), and returns; the
 * call's output is undefined.  Applies to launches made after the call, from
 * any thread; not for production use.  Returns PKV_ERR_INVALID_ARG above the
 * default. */
pkv_status pkv_testing_set_handoff_wait_ns(unsigned long long ns);

const char *pkv_status_str(pkv_status s);

/* ABI version: (major << 16) | minor. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
