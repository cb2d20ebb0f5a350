// pkv_noalloc.cu -- paged_decode_attn for callers that cannot allocate.
//
// Some callers cannot hand the library a workspace: code that runs where
// cudaMalloc is off limits (inside a memory-pool-managed runtime that owns
// every device allocation, in a plugin host that forbids allocation during
// its execute phase, or on a path that must never fail on out-of-memory).
// For them this file keeps the workspace in a file-scope device array of
// fixed size.  Every GPU that loads this library holds the array until the
// process exits; the entry point itself calls no allocator.
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

// The scratch: header (status word first), row bookkeeping and partials, laid
// out exactly like a caller-owned workspace of pkv_workspace_bytes() bytes.
static __device__ __align__(256) unsigned char g_pkv_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device

// In host code g_pkv_noalloc_scratch names a host-side stand-in, not device
// memory: the device address must come from cudaGetSymbolAddress, asked
// once per device with that device current.
pkv_status scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PKV_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_noalloc_scratch) != cudaSuccess || p == nullptr)
            return PKV_ERR_LAUNCH;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

} // namespace

extern "C" pkv_status paged_decode_attn_noalloc(const pkv_dims *dims, const void *q,
                                                const void *k_pool, const void *v_pool,
                                                const int32_t *kv_indices,
                                                const int32_t *kv_indptr,
                                                const int32_t *seq_lens, int num_splits,
                                                void *out, uint32_t *status,
                                                pkv_stream_t stream)
{
    // the shape checks of paged_decode_attn, with its status codes
    const pkv_status dst = pkv::check_dims(dims);
    if (dst != PKV_OK)
        return dst;
    if (num_splits < 1 || num_splits > pkv::kMaxSplits)
        return PKV_ERR_INVALID_ARG;
    if (pkv_workspace_bytes(dims, num_splits) > PKV_NOALLOC_SCRATCH_BYTES)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3) != 0)
        return PKV_ERR_INVALID_ARG;
    if (dims->B == 0) {
        // nothing to compute, but the caller's status word still starts this
        // call at zero
        if (status != nullptr &&
            cudaMemsetAsync(status, 0, sizeof(uint32_t), (cudaStream_t)stream) != cudaSuccess)
            return PKV_ERR_LAUNCH;
        return PKV_OK;
    }
    void *scratch = nullptr;
    pkv_status st = scratch_for_current_device(&scratch);
    if (st != PKV_OK)
        return st;
    // the status word must start at zero; the rest is written before it is read
    if (cudaMemsetAsync(scratch, 0, 256, (cudaStream_t)stream) != cudaSuccess)
        return PKV_ERR_LAUNCH;
    st = paged_decode_attn(dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, num_splits,
                           scratch, PKV_NOALLOC_SCRATCH_BYTES, out, stream);
    if (st != PKV_OK || status == nullptr)
        return st;
    return cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                           (cudaStream_t)stream) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_LAUNCH;
}
