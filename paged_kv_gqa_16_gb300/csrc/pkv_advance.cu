// pkv_advance.cu -- decode metadata on the device: the advance (one more
// token per live row, and a page from the free list for each row whose new
// token starts a page), and the one-page-per-row table of a contiguous cache.
//
// What it computes (AstrAI commit log, compare v1.3.12..6f09b1d,
// astrai/inference/core/cache.py): PagePool.task_extend(pos) claims the slot
// of position pos, and _extend_slot takes a fresh page from the allocator
// when pos / page_size is past the row's pages, then the length becomes
// pos + 1; in the steady state bind_tasks adds one to every row's length in
// place.  Here pos = seq_lens[b] for every row with seq_lens[b] > 0, and the
// allocator is a device free list consumed in row order.
//
// Layout of the work: one block (advance_block, pkv_advance.cuh): its
// threads walk the rows a block at a time.  Each thread decides for its row
// whether it wants a page; a block scan of those wants gives each row its
// rank, so row b takes free_pages[head + rank], the same assignment a
// sequential walk in increasing b makes.  Each thread reads and writes only
// its own row.  The same block also runs inside the piece combine of
// paged_decode_step_advance.
#include "pkv_advance.cuh"

namespace pkv {

namespace {

constexpr int kAdvanceThreads = 1024;

__global__ void __launch_bounds__(kAdvanceThreads) advance_kernel(const AdvanceParams p)
{
    // the lengths may come from the step just before; the next step's decode
    // may start its prologue and waits for this grid before reading them
    grid_dependency_wait();
    grid_launch_dependents();
    advance_block(p);
}

// A contiguous cache [num_slots, cache_len, Hkv, D] read through cache_batch_idx
// (compare v1.3.12..6f09b1d, attention_backend.py: "Read K/V directly from
// flat pool via cache_batch_idx + cache_seqlens") is a paged pool whose pages
// are cache_len tokens long, with one page per row: row b's table is
// {cache_batch_idx[b]}.
__global__ void __launch_bounds__(256) contig_table_kernel(const int32_t *idx, int B,
                                                           int32_t *table)
{
    grid_dependency_wait();
    grid_launch_dependents();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= B; i += gridDim.x * blockDim.x) {
        table[i] = i;                                 // kv_indptr
        if (i < B)
            table[B + 1 + i] = idx != nullptr ? idx[i] : i;
    }
}

} // namespace

cudaError_t launch_contig_table(const int32_t *idx, int B, int32_t *table, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    const int blocks = (B + 1 + 255) / 256;
    cfg.gridDim = dim3(blocks < 64 ? blocks : 64);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, contig_table_kernel, idx, B, table);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

cudaError_t launch_advance(const AdvanceParams &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kAdvanceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, advance_kernel, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace pkv
