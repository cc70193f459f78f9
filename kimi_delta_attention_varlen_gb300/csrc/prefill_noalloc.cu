// kda_prefill_varlen_noalloc: the chunked prefill for callers that cannot
// allocate device memory.
//
// kda_prefill_varlen needs a caller-provided workspace.  Some callers cannot
// provide one: a C or C++ host program that links only this library and has
// no device allocator of its own; a serving runtime that fixes its device
// memory budget at start-up and forbids allocations on the request path
// (cudaMalloc can synchronise the device and can fail once memory is
// fragmented); code that must not call into an allocator while work is in
// flight.  For them, this entry point runs the very same kernels with the
// workspace placed in a fixed array of device memory owned by this library.
//
// The array is a file-scope __device__ variable of KDA_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU that loads the library holds it until the process exits.
// Its device address is looked up once per device, with that device current,
// on the first call made on that device (so make that first call before any
// stream capture).  All calls share the one array: calls that overlap on the
// GPU (on different streams, or from different threads without ordering) race
// and corrupt each other's results.  Nothing in the array needs clearing
// between calls: every byte the kernels read is written earlier in the same
// call (the chunk table kernel resets the status word at the array's start).
// kda_prefill_noalloc_status reads that status word.  No function here
// allocates.
#include <cuda_runtime.h>

#include <mutex>

#include "kda_internal.h"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;

// Device memory.  Host code must never dereference this name or take its
// address for use as a pointer (on the host it names a shadow variable, not
// the device array); the device address comes only from cudaGetSymbolAddress
// in scratch_address below, cached per device.
__device__ __align__(256) char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the device current to this thread.
cudaError_t scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int kda_prefill_varlen_noalloc(const void *q, const void *k, const void *v, int32_t io_dtype,
                                          const float *g, const float *beta, const int32_t *cu_seqlens,
                                          int64_t num_seqs, int64_t total_tokens, int32_t h, int32_t dk, int32_t dv,
                                          float scale, int32_t qk_l2norm, const void *init_state,
                                          int32_t init_dtype, float *final_state, void *out, void *stream)
{
    // the compact form (bf16, head size 128) needs no per-chunk records
    const size_t need = kda_prefill_workspace_size_compact(total_tokens, num_seqs, h, dk, dv, io_dtype);
    if (need > kScratchBytes) return KDA_ERR_WORKSPACE;  // batch too large for the fixed scratch
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return kda::record_cuda_status(e);
    return kda_prefill_varlen(q, k, v, io_dtype, g, beta, cu_seqlens, num_seqs, total_tokens, h, dk, dv, scale,
                              qk_l2norm, init_state, init_dtype, final_state, out, scratch, kScratchBytes, stream);
}

extern "C" int kda_prefill_noalloc_status(int32_t *status_out, void *stream)
{
    if (status_out == nullptr) return KDA_ERR_NULL;
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return kda::record_cuda_status(e);
    return kda_prefill_workspace_status(scratch, status_out, stream);
}
