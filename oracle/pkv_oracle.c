/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or table with the CUDA path.
 *
 * What it computes, and where the pages define it.  The pages are the AstrAI
 * commit log: "compare v1.3.12..6f09b1d" (a unified diff; files named below
 * are hunks of it), "commits by author" (a listing of commit messages) and
 * "commit 0573962: astrai/inference".
 *
 *   - compare v1.3.12..6f09b1d, astrai/extension/attention_ops.py, docstring
 *       of attn_paged_decode: a packed [batch, n_heads, head_dim] query
 *       attends over the K/V rows of its request, gathered from a pool
 *       through a table; output [batch, n_heads, head_dim].  The removed
 *       lines of the same hunk give the paged pool layout
 *       [n_pages, page_size, n_kv_heads, head_dim] addressed by a page table.
 *   - same diff, astrai/extension/attention_backend.py,
 *       TorchNativeBackend.fwd_decode: gather by table, repeat_kv(n_rep)
 *       (query head h reads kv head h / n_rep), then
 *       scaled_dot_product_attention = softmax(q K^T / sqrt(D)) V.
 *   - same diff, astrai/inference/core/cache.py, PagePool._extend_slot: the
 *       slot of logical position pos is page_table[pos / page_size] *
 *       page_size + pos % page_size; task_extend sets the length to pos + 1
 *       and bind_tasks writes the new token at seq_len - 1.
 *   - commits by author, "Fix rotary docs to describe cos/sin freqs_cis
 *       table" and "apply_rotary_emb ... torch complex multiply path": RoPE
 *       multiplies each interleaved pair x[2i] + j x[2i+1] by
 *       exp(j * pos * theta_i).
 *   - commits by author, split-KV decode ("split partials", "single combine
 *       kernel", "compute_num_splits"): per-split partial outputs and
 *       (max, sum) statistics merged by a combine pass.
 *   - the same appends for a chunk of tokens per row (po_extend).
 *   - same diff, attention_ops.py, attn_paged_prefill / attn_prefill: a
 *       ragged chunk of queries per request, the last of its tokens, each
 *       attending causally up to its own position (po_prefill).
 *   - same diff, cache.py, PagePool.task_extend / _extend_slot and the
 *       steady-state branch of bind_tasks: one more token per task, and a
 *       page from the allocator when the token starts a page (po_advance).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - kv_indptr[b] .. kv_indptr[b+1] indexes the PAGES of row b in kv_indices;
 *     seq_lens[b] counts tokens, including the token appended this step.
 *   - theta_i = base^(-2i/D), i in [0, D/2); position of the new token = L-1.
 *   - a row with seq_len 0 produces an all-zero output.
 *   - split s of a row covers logical tokens [s*chunk, min((s+1)*chunk, L));
 *     an empty split has m = -inf, l = 0.
 *   - ml holds (m, l): m = max score, l = sum exp(score - m); o_part is
 *     normalised (divided by l).
 *
 * All arithmetic is IEEE double; bf16 inputs are widened exactly.  Rounding
 * back to bf16 (append only) is round-to-nearest-even, done once from double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PO_OK 0
#define PO_ERR (-1)

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double po_bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even, in ONE rounding
 * (no detour through binary32, which would round twice).  bf16 has an 8-bit
 * significand (7 stored bits) and binary32's exponent range, so:
 *   - normal range |x| >= 2^-126: the spacing in the binade [2^(E-1), 2^E) is
 *     2^(E-8); scale by its inverse (exact), round to an integer with
 *     nearbyint (ties-to-even in the default rounding mode), scale back;
 *   - below 2^-126 the spacing is the fixed subnormal step 2^-133.
 * The result is a bf16 value (or +-inf on overflow), exactly representable in
 * binary32, whose upper 16 bits are the encoding. */
uint16_t po_f64_to_bf16_rne(double x)
{
    if (isnan(x))
        return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    double r;
    if (x == 0.0 || isinf(x)) {
        r = x;
    } else if (fabs(x) < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(x, 133)), -133);
    } else {
        int e;
        (void)frexp(x, &e);                /* |x| in [2^(e-1), 2^e) */
        r = ldexp(nearbyint(ldexp(x, 8 - e)), e - 8);
    }
    float f = (float)r;                    /* exact, or +-inf past the range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void po_f64_to_bf16_array(const double *x, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = po_f64_to_bf16_rne(x[i]);
}

void po_bf16_to_f64_array(const uint16_t *x, double *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = po_bf16_to_f64(x[i]);
}

/* ---------------------------------------------------------------- RoPE -- */

/* Rotate one head vector x[0..D) by position pos: pair i = (x[2i], x[2i+1])
 * is multiplied, as a complex number x[2i] + j x[2i+1], by
 * exp(j * pos * theta_i) with theta_i = base^(-2i/D). */
void po_rope_rotate(const double *x, double *y, int D, long pos, double base)
{
    for (int i = 0; i < D / 2; ++i) {
        double theta = pow(base, -2.0 * (double)i / (double)D);
        double ang = (double)pos * theta;
        double c = cos(ang), s = sin(ang);
        double a = x[2 * i], b = x[2 * i + 1];
        y[2 * i] = a * c - b * s;
        y[2 * i + 1] = a * s + b * c;
    }
}

/* ------------------------------------------------------------ indexing -- */

/* Element offset of (page, slot, kv head g, d = 0) in a pool laid out as
 * [num_pages, page_size, Hkv, D]. */
static long pool_offset(long page, long slot, int g, int page_size, int Hkv, int D)
{
    return ((page * page_size + slot) * Hkv + g) * (long)D;
}

/* Physical (page, slot) of logical token t of row b; -1 if the table does not
 * hold it or names a page outside the pool. */
static int locate(int b, long t, int page_size, int num_pages,
                  const int32_t *kv_indices, const int32_t *kv_indptr,
                  long *page, long *slot)
{
    long pi = t / page_size;
    long n_row_pages = (long)kv_indptr[b + 1] - (long)kv_indptr[b];
    if (t < 0 || pi >= n_row_pages)
        return PO_ERR;
    long p = kv_indices[kv_indptr[b] + pi];
    if (p < 0 || p >= num_pages)
        return PO_ERR;
    *page = p;
    *slot = t % page_size;
    return PO_OK;
}

/* Logically ordered K and V rows of (row b, kv head g): outK/outV [L, D]. */
int po_gather(int b, int g, int Hkv, int D, int page_size, int num_pages,
              const uint16_t *k_pool, const uint16_t *v_pool,
              const int32_t *kv_indices, const int32_t *kv_indptr,
              const int32_t *seq_lens, double *outK, double *outV)
{
    long L = seq_lens[b];
    for (long t = 0; t < L; ++t) {
        long page, slot;
        if (locate(b, t, page_size, num_pages, kv_indices, kv_indptr, &page, &slot))
            return PO_ERR;
        long off = pool_offset(page, slot, g, page_size, Hkv, D);
        for (int d = 0; d < D; ++d) {
            outK[t * D + d] = po_bf16_to_f64(k_pool[off + d]);
            outV[t * D + d] = po_bf16_to_f64(v_pool[off + d]);
        }
    }
    return PO_OK;
}

/* -------------------------------------------------------------- append -- */

/* Write each row's new token into its slot.  For row b with L = seq_lens[b]
 * > 0, the token sits at logical position p = L - 1; its K head vectors are
 * rotated by p (if use_rope) and rounded to bf16, V is copied unchanged.  If
 * rope_q, every query head of the row is rotated by p in place.  Rows with
 * L = 0 are skipped. */
int po_append(int B, int Hq, int Hkv, int D, int page_size, int num_pages,
              uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
              uint16_t *k_pool, uint16_t *v_pool,
              const int32_t *kv_indices, const int32_t *kv_indptr,
              const int32_t *seq_lens, int use_rope, double rope_base, int rope_q)
{
    double *x = malloc(sizeof(double) * (size_t)D);
    double *y = malloc(sizeof(double) * (size_t)D);
    int rc = PO_OK;
    for (int b = 0; b < B && rc == PO_OK; ++b) {
        long L = seq_lens[b];
        if (L <= 0)
            continue;
        long p = L - 1, page, slot;
        if (locate(b, p, page_size, num_pages, kv_indices, kv_indptr, &page, &slot)) {
            rc = PO_ERR;
            break;
        }
        for (int g = 0; g < Hkv; ++g) {
            const uint16_t *kin = k_new + ((long)b * Hkv + g) * D;
            const uint16_t *vin = v_new + ((long)b * Hkv + g) * D;
            long off = pool_offset(page, slot, g, page_size, Hkv, D);
            for (int d = 0; d < D; ++d)
                x[d] = po_bf16_to_f64(kin[d]);
            if (use_rope)
                po_rope_rotate(x, y, D, p, rope_base);
            else
                memcpy(y, x, sizeof(double) * (size_t)D);
            for (int d = 0; d < D; ++d) {
                k_pool[off + d] = po_f64_to_bf16_rne(y[d]);
                v_pool[off + d] = vin[d];
            }
        }
        if (use_rope && rope_q) {
            for (int h = 0; h < Hq; ++h) {
                uint16_t *qh = q + ((long)b * Hq + h) * D;
                for (int d = 0; d < D; ++d)
                    x[d] = po_bf16_to_f64(qh[d]);
                po_rope_rotate(x, y, D, p, rope_base);
                for (int d = 0; d < D; ++d)
                    qh[d] = po_f64_to_bf16_rne(y[d]);
            }
        }
    }
    free(x);
    free(y);
    return rc;
}

/* ------------------------------------------------------------- softmax -- */

/* Attention of one query vector qv[D] over tokens [t0, t1) of (b, g):
 *   s_t = scale * <q, k_t>,  m = max s_t,  l = sum exp(s_t - m),
 *   o   = sum exp(s_t - m) v_t / l.
 * Returns the number of tokens; with none, m = -inf, l = 0 and o = 0. */
static long attend_range(const double *qv, int b, int g, long t0, long t1,
                         int Hkv, int D, int page_size, int num_pages,
                         const uint16_t *k_pool, const uint16_t *v_pool,
                         const int32_t *kv_indices, const int32_t *kv_indptr,
                         double scale, double *s_buf, double *o, double *m_out,
                         double *l_out, int *err)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (t1 <= t0)
        return 0;
    double m = -INFINITY;
    for (long t = t0; t < t1; ++t) {
        long page, slot;
        if (locate(b, t, page_size, num_pages, kv_indices, kv_indptr, &page, &slot)) {
            *err = 1;
            return 0;
        }
        const uint16_t *k = k_pool + pool_offset(page, slot, g, page_size, Hkv, D);
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += qv[d] * po_bf16_to_f64(k[d]);
        s_buf[t - t0] = scale * acc;
        if (s_buf[t - t0] > m)
            m = s_buf[t - t0];
    }
    double l = 0.0;
    for (long t = t0; t < t1; ++t) {
        long page = 0, slot = 0;   /* every t was located in the first pass */
        locate(b, t, page_size, num_pages, kv_indices, kv_indptr, &page, &slot);
        const uint16_t *v = v_pool + pool_offset(page, slot, g, page_size, Hkv, D);
        double p = exp(s_buf[t - t0] - m);
        l += p;
        for (int d = 0; d < D; ++d)
            o[d] += p * po_bf16_to_f64(v[d]);
    }
    for (int d = 0; d < D; ++d)
        o[d] /= l;
    *m_out = m;
    *l_out = l;
    return t1 - t0;
}

static long max_len(int B, const int32_t *seq_lens)
{
    long mx = 0;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] > mx)
            mx = seq_lens[b];
    return mx;
}

/* Extend: write a chunk of new tokens per row, the multi-token form of
 * po_append (compare v1.3.12..6f09b1d, attention_backend.py: the prefill path
 * stores every new token's K/V at its slot, k_buffer[layer, out_cache_loc];
 * cache.py: the slot of position pos is page_table[pos / page_size] *
 * page_size + pos % page_size).  Row b's q_len = qo_indptr[b+1] -
 * qo_indptr[b] tokens are the last q_len of its L = seq_lens[b]: token i
 * (input row qo_indptr[b] + i) sits at position L - q_len + i.  K is rotated
 * by that position (when use_rope), V copied; with rope_q the token's query
 * heads are rotated the same way, in place.  A row with q_len < 0 or > L, or
 * a qo_indptr that does not walk from 0 to total_q, is an error. */
int po_extend(int B, int Hq, int Hkv, int D, int page_size, int num_pages, int total_q,
              uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
              const int32_t *qo_indptr, uint16_t *k_pool, uint16_t *v_pool,
              const int32_t *kv_indices, const int32_t *kv_indptr, const int32_t *seq_lens,
              int use_rope, double rope_base, int rope_q)
{
    if (qo_indptr[0] != 0 || qo_indptr[B] != total_q)
        return PO_ERR;
    double *x = malloc(sizeof(double) * (size_t)D);
    double *y = malloc(sizeof(double) * (size_t)D);
    int rc = PO_OK;
    for (int b = 0; b < B && rc == PO_OK; ++b) {
        const long L = seq_lens[b];
        const long q_len = (long)qo_indptr[b + 1] - qo_indptr[b];
        if (q_len < 0 || q_len > L) {
            rc = PO_ERR;
            break;
        }
        for (long i = 0; i < q_len && rc == PO_OK; ++i) {
            const long t = qo_indptr[b] + i;
            const long pos = L - q_len + i;
            long page, slot;
            if (locate(b, pos, page_size, num_pages, kv_indices, kv_indptr, &page, &slot)) {
                rc = PO_ERR;
                break;
            }
            for (int g = 0; g < Hkv; ++g) {
                const uint16_t *kin = k_new + (t * Hkv + g) * D;
                const uint16_t *vin = v_new + (t * Hkv + g) * D;
                const long off = pool_offset(page, slot, g, page_size, Hkv, D);
                for (int d = 0; d < D; ++d)
                    x[d] = po_bf16_to_f64(kin[d]);
                if (use_rope)
                    po_rope_rotate(x, y, D, pos, rope_base);
                else
                    memcpy(y, x, sizeof(double) * (size_t)D);
                for (int d = 0; d < D; ++d) {
                    k_pool[off + d] = po_f64_to_bf16_rne(y[d]);
                    v_pool[off + d] = vin[d];
                }
            }
            if (use_rope && rope_q) {
                for (int h = 0; h < Hq; ++h) {
                    uint16_t *qh = q + (t * Hq + h) * D;
                    for (int d = 0; d < D; ++d)
                        x[d] = po_bf16_to_f64(qh[d]);
                    po_rope_rotate(x, y, D, pos, rope_base);
                    for (int d = 0; d < D; ++d)
                        qh[d] = po_f64_to_bf16_rne(y[d]);
                }
            }
        }
    }
    free(x);
    free(y);
    return rc;
}

/* out[b, h, :] = softmax(q[b,h] K_{b,g}^T * scale) V_{b,g}, g = h / (Hq/Hkv),
 * over the L = seq_lens[b] logically ordered rows; zero where L = 0.
 * out is [B, Hq, D] doubles. */
int po_decode(int B, int Hq, int Hkv, int D, int page_size, int num_pages,
              const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
              const int32_t *kv_indices, const int32_t *kv_indptr,
              const int32_t *seq_lens, double scale, double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return PO_ERR;
    int n_rep = Hq / Hkv;
    long Lmax = max_len(B, seq_lens);
    int err = 0;
#pragma omp parallel
    {
        double *qv = malloc(sizeof(double) * (size_t)D);
        double *s = malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
#pragma omp for collapse(2) schedule(dynamic)
        for (int b = 0; b < B; ++b) {
            for (int h = 0; h < Hq; ++h) {
                int g = h / n_rep, e = 0;
                double m, l;
                const uint16_t *qh = q + ((long)b * Hq + h) * D;
                for (int d = 0; d < D; ++d)
                    qv[d] = po_bf16_to_f64(qh[d]);
                attend_range(qv, b, g, 0, seq_lens[b], Hkv, D, page_size, num_pages,
                             k_pool, v_pool, kv_indices, kv_indptr, scale, s,
                             out + ((long)b * Hq + h) * D, &m, &l, &e);
                if (e) {
#pragma omp atomic write
                    err = 1;
                }
            }
        }
        free(qv);
        free(s);
    }
    return err ? PO_ERR : PO_OK;
}

/* Prefill / extend over the paged pool (compare v1.3.12..6f09b1d,
 * astrai/extension/attention_ops.py, docstring of attn_paged_prefill: a
 * ragged batch, q [total_q, n_heads, head_dim] flattened across requests,
 * qo_indptr the prefix sum of the requests' query lengths, causal; and
 * attn_prefill, whose causal offset is kv_len - q_len).  Row b's
 * q_len = qo_indptr[b+1] - qo_indptr[b] queries are the last q_len of its
 * L = seq_lens[b] tokens, so query i sits at position L - q_len + i and
 * attends keys 0 .. that position.  out [total_q, Hq, D] doubles.  A row
 * with q_len > L, or a qo_indptr that is not a non-decreasing walk from 0
 * to total_q, is an error. */
int po_prefill(int B, int Hq, int Hkv, int D, int page_size, int num_pages, int total_q,
               const uint16_t *q, const int32_t *qo_indptr, const uint16_t *k_pool,
               const uint16_t *v_pool, const int32_t *kv_indices, const int32_t *kv_indptr,
               const int32_t *seq_lens, double scale, double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || qo_indptr[0] != 0 || qo_indptr[B] != total_q)
        return PO_ERR;
    int *row_of = malloc(sizeof(int) * (size_t)(total_q > 0 ? total_q : 1));
    for (int b = 0; b < B; ++b) {
        const int q_len = qo_indptr[b + 1] - qo_indptr[b];
        if (q_len < 0 || q_len > seq_lens[b]) {
            free(row_of);
            return PO_ERR;
        }
        for (int i = qo_indptr[b]; i < qo_indptr[b + 1]; ++i)
            row_of[i] = b;
    }
    const int n_rep = Hq / Hkv;
    const long Lmax = max_len(B, seq_lens);
    int err = 0;
#pragma omp parallel
    {
        double *qv = malloc(sizeof(double) * (size_t)D);
        double *s = malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
#pragma omp for collapse(2) schedule(dynamic)
        for (int i = 0; i < total_q; ++i) {
            for (int h = 0; h < Hq; ++h) {
                const int b = row_of[i];
                const long pos = (long)seq_lens[b] - (qo_indptr[b + 1] - qo_indptr[b]) +
                                 (i - qo_indptr[b]);
                int e = 0;
                double m, l;
                const uint16_t *qh = q + ((long)i * Hq + h) * D;
                for (int d = 0; d < D; ++d)
                    qv[d] = po_bf16_to_f64(qh[d]);
                attend_range(qv, b, h / n_rep, 0, pos + 1, Hkv, D, page_size, num_pages,
                             k_pool, v_pool, kv_indices, kv_indptr, scale, s,
                             out + ((long)i * Hq + h) * D, &m, &l, &e);
                if (e) {
#pragma omp atomic write
                    err = 1;
                }
            }
        }
        free(qv);
        free(s);
    }
    free(row_of);
    return err ? PO_ERR : PO_OK;
}

/* Split partials: split s of row b covers tokens [s*chunk, min((s+1)*chunk, L)).
 * o_part [B, Hq, S, D] holds the split's normalised output, ml_part
 * [B, Hq, S, 2] its (m, l).  Splits past the row's end are empty. */
int po_decode_partials(int B, int Hq, int Hkv, int D, int page_size, int num_pages,
                       const uint16_t *q, const uint16_t *k_pool,
                       const uint16_t *v_pool, const int32_t *kv_indices,
                       const int32_t *kv_indptr, const int32_t *seq_lens,
                       double scale, int num_splits, long chunk,
                       double *o_part, double *ml_part)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || num_splits <= 0 || chunk <= 0)
        return PO_ERR;
    int n_rep = Hq / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double *qv = malloc(sizeof(double) * (size_t)D);
        double *s = malloc(sizeof(double) * (size_t)chunk);
#pragma omp for collapse(2) schedule(dynamic)
        for (int b = 0; b < B; ++b) {
            for (int h = 0; h < Hq; ++h) {
                int g = h / n_rep;
                const uint16_t *qh = q + ((long)b * Hq + h) * D;
                for (int d = 0; d < D; ++d)
                    qv[d] = po_bf16_to_f64(qh[d]);
                for (int sp = 0; sp < num_splits; ++sp) {
                    long t0 = (long)sp * chunk, t1 = t0 + chunk;
                    if (t1 > seq_lens[b])
                        t1 = seq_lens[b];
                    long slot = ((long)b * Hq + h) * num_splits + sp;
                    int e = 0;
                    attend_range(qv, b, g, t0, t1, Hkv, D, page_size, num_pages,
                                 k_pool, v_pool, kv_indices, kv_indptr, scale, s,
                                 o_part + slot * D, &ml_part[2 * slot],
                                 &ml_part[2 * slot + 1], &e);
                    if (e) {
#pragma omp atomic write
                        err = 1;
                    }
                }
            }
        }
        free(qv);
        free(s);
    }
    return err ? PO_ERR : PO_OK;
}

/* Merge S partials of each (b, h): M = max over non-empty splits of m_s,
 * w_s = l_s exp(m_s - M), out = sum_s w_s o_s / sum_s w_s.  Splits with
 * l_s = 0 contribute nothing; if every split is empty the output is 0.
 * o_part [B, Hq, S, D], ml_part [B, Hq, S, 2], out [B, Hq, D], all double
 * (the library's binary32 partials widen exactly). */
int po_combine(int B, int Hq, int D, int num_splits, const double *o_part,
               const double *ml_part, double *out)
{
    if (num_splits <= 0)
        return PO_ERR;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            long base = ((long)b * Hq + h) * num_splits;
            double *o = out + ((long)b * Hq + h) * D;
            double M = -INFINITY;
            for (int s = 0; s < num_splits; ++s)
                if (ml_part[2 * (base + s) + 1] > 0.0 && ml_part[2 * (base + s)] > M)
                    M = ml_part[2 * (base + s)];
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            double den = 0.0;
            for (int s = 0; s < num_splits; ++s) {
                double l = ml_part[2 * (base + s) + 1];
                if (!(l > 0.0))
                    continue;
                double w = l * exp(ml_part[2 * (base + s)] - M);
                den += w;
                for (int d = 0; d < D; ++d)
                    o[d] += w * o_part[(base + s) * D + d];
            }
            if (den > 0.0)
                for (int d = 0; d < D; ++d)
                    o[d] /= den;
        }
    }
    return PO_OK;
}

/* ------------------------------------------------------------- threads -- */

/* ------------------------------------------------------------- advance -- */

/* One steady-state decode step of metadata, in the pages' order (compare
 * v1.3.12..6f09b1d, astrai/inference/core/cache.py: PagePool.task_extend
 * refuses pos >= max_seq_len; _extend_slot computes page_idx = pos /
 * page_size and, when that is past the pages the task holds, takes a page
 * from the allocator, failing if it has none; task_extend then sets the
 * length to pos + 1).  The tasks are the rows with seq_lens[b] > 0, visited
 * in increasing b; the new token's position is pos = seq_lens[b]; the pages
 * a row holds are ceil(pos / page_size), so page_idx is past them exactly
 * when pos is a multiple of page_size; the allocator hands out
 * free_pages[*head], free_pages[*head + 1], ... in the order of the calls.
 * A row's page list lives at kv_indices[kv_indptr[b] ...] with room for
 * kv_indptr[b+1] - kv_indptr[b] entries; a row with no room, or one that
 * finds the list empty, keeps its length.
 * Counts the rows refused for length (*n_len) and for want of a page or an
 * entry (*n_page); rows whose kv_indptr pair is malformed count in *n_bad.
 * Returns 0. */
int po_advance(int B, int page_size, int max_seq_len, int num_indices, int32_t *seq_lens,
               const int32_t *kv_indptr, int32_t *kv_indices, const int32_t *free_pages,
               int num_free, int32_t *head, int *n_len, int *n_page, int *n_bad)
{
    *n_len = *n_page = *n_bad = 0;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        if (L <= 0)
            continue;                       /* not a task this step */
        const int pos = L;
        if (pos >= max_seq_len) {
            ++*n_len;
            continue;
        }
        const int page_idx = pos / page_size;
        const int held = (L + page_size - 1) / page_size;
        if (page_idx >= held) {             /* the token starts a new page */
            const int first = kv_indptr[b], room = kv_indptr[b + 1] - kv_indptr[b];
            if (first < 0 || room < 0 || kv_indptr[b + 1] > num_indices) {
                ++*n_bad;
                continue;
            }
            if (page_idx >= room || *head >= num_free) {
                ++*n_page;
                continue;
            }
            kv_indices[first + page_idx] = free_pages[*head];
            ++*head;
        }
        seq_lens[b] = pos + 1;
    }
    return 0;
}

void po_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int po_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
