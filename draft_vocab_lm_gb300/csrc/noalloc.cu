// dvl_draft_argmax_noalloc: draft_argmax without a caller-supplied workspace.
//
// Some callers cannot allocate device memory for the reduction workspace:
// code that runs as a plugin inside an inference engine which owns every
// device allocation (its allocator accounts for and pools all memory, and
// raw cudaMalloc is not available to plugins), and latency-critical decode
// loops where a cudaMalloc would stall the pipeline (it may synchronize the
// device and takes far longer than the call itself).  For them this entry
// point keeps its scratch in a fixed array in the library's own device
// memory, so the caller passes only the head, the hidden rows and the
// outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "dvl.h"
#include "dvl_internal.h"

namespace {

// The scratch: the cross-block reduction state of one argmax call with up
// to DVL_MAX_M hidden rows (ticket, status word, one best key per row).
// Every GPU that loads the library holds these bytes until the process
// exits.
constexpr size_t kScratchBytes = dvl::kWsSlots;  // 512 bytes
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_ptr[kMaxDevices] = {};

// The array's device address on the current device.  Host code may not use
// g_noalloc_scratch itself: on the host that name is only a stand-in.
dvl_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return DVL_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return DVL_ERR_CUDA;
        g_ptr[dev] = p;
    }
    *out = g_ptr[dev];
    return DVL_OK;
}

}  // namespace

extern "C" dvl_status dvl_draft_argmax_noalloc(const dvl_head *head, const void *h, int32_t M,
                                               int32_t *ids, float *max_logit, void *stream)
{
    if (M < 1 || M > DVL_MAX_M)
        return DVL_ERR_INVALID_ARG;  // beyond what the fixed scratch holds
    if (dvl_workspace_bytes(M, 1) > kScratchBytes)
        return DVL_ERR_WORKSPACE;
    dvl_status chk = dvl::check_reduce_args(head, h, M, 1, ids, max_logit);
    if (chk != DVL_OK)
        return chk;  // nothing enqueued
    void *scratch = nullptr;
    dvl_status st = scratch_address(&scratch);
    if (st != DVL_OK)
        return st;
    // The reduction state must start at zero; clear it in stream order.
    if (cudaMemsetAsync(scratch, 0, kScratchBytes, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return DVL_ERR_CUDA;
    return dvl_draft_argmax(head, h, M, ids, max_logit, scratch, kScratchBytes, stream);
}
