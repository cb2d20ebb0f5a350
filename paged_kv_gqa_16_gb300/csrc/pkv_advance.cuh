// pkv_advance.cuh -- the decode metadata advance as the work of one block,
// shared by its own kernel and the piece combine of the fused step.
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// One block of blockDim.x threads (a multiple of 32, at most 1024) advances
// every row: one more token for each row with seq_lens[b] > 0, and, for a
// row whose new token starts a page, the next free page in increasing row
// order (a ballot and block scan rank the rows that want one).  Refused rows
// keep their length and raise a flag.  Every thread of the block calls it.
__device__ __forceinline__ void advance_block(const AdvanceParams &p)
{
    constexpr unsigned kAllLanes = 0xffffffffu;
    __shared__ int s_warp[32];
    __shared__ unsigned s_flags;
    const int nthr = blockDim.x, nwarp = nthr >> 5;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0)
        s_flags = 0u;
    const int head = *p.free_head;
    int taken = 0;                                    // wants in earlier chunks
    unsigned flags = 0u;
    for (int base = 0; base < p.B; base += nthr) {
        const int b = base + (int)threadIdx.x;
        const int L = b < p.B ? p.seq_lens[b] : 0;
        const int pos = L;
        bool advance = L > 0;
        bool want = false;
        int slot = -1;
        if (advance && pos >= p.max_seq_len) {
            flags |= kFlagBadLen;
            advance = false;
        }
        if (advance && pos % p.page_size == 0) {
            const int pg0 = p.kv_indptr[b], pg1 = p.kv_indptr[b + 1];
            const int idx = pos / p.page_size;
            if (pg0 < 0 || pg1 < pg0 || pg1 > p.num_indices) {
                flags |= kFlagBadPage;
                advance = false;
            } else if (idx >= pg1 - pg0) {
                flags |= kFlagNoPage;                 // the row's table is full
                advance = false;
            } else {
                want = true;
                slot = pg0 + idx;
            }
        }
        // exclusive scan of the wants over the chunk, in row order
        const unsigned bal = __ballot_sync(kAllLanes, want);
        const int in_warp = __popc(bal & ((1u << lane) - 1u));
        if (lane == 0)
            s_warp[warp] = __popc(bal);
        __syncthreads();
        int before = 0, chunk_total = 0;
        for (int w = 0; w < nwarp; ++w) {
            const int c = s_warp[w];
            before += w < warp ? c : 0;
            chunk_total += c;
        }
        __syncthreads();                              // s_warp is rewritten next chunk
        if (want) {
            const long long k = (long long)head + taken + before + in_warp;
            if (k < p.num_free) {
                p.kv_indices[slot] = p.free_pages[k];
            } else {
                flags |= kFlagNoPage;                 // the free list ran out
                advance = false;
            }
        }
        if (advance)
            p.seq_lens[b] = pos + 1;
        taken += chunk_total;
    }
    if (flags != 0u)
        atomicOr(&s_flags, flags);
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long left = (long long)p.num_free - head;
        const long long got = taken < left ? taken : (left > 0 ? left : 0);
        *p.free_head = head + (int)got;
        if (s_flags != 0u && p.status != nullptr)
            atomicOr(p.status, s_flags);
    }
}

} // namespace pkv
