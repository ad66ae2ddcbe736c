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
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>

#include "dvl.h"
#include "dvl_internal.h"

namespace {

// The scratch: the cross-block reduction state of one argmax call with up
// to DVL_MAX_M hidden rows (ticket, status word, one best key per row), laid
// out like a workspace.  Every GPU that loads the library holds these bytes
// until the process exits.
constexpr size_t kScratchBytes = dvl::kWsSlots;  // 512 bytes
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// The array's device address, per CUDA context.  A context id (cuCtxGetId)
// is never reused within a process, so an address looked up before a
// context was torn down (cudaDeviceReset) is never handed out again.
std::mutex g_mu;
std::map<unsigned long long, void *> g_ptr;

struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};

// The driver's context queries through the runtime's entry-point lookup (no
// link against the driver library).
const CtxFns &ctx_fns()
{
    static std::once_flag once;
    static CtxFns f;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    return f;
}

// Id of the calling thread's current context; false if there is none yet or
// the driver cannot say.
bool current_ctx_id(unsigned long long *id)
{
    const CtxFns &f = ctx_fns();
    if (!f.get_current || !f.get_id)
        return false;
    CUcontext c = nullptr;
    if (f.get_current(&c) != CUDA_SUCCESS || !c)
        return false;
    return f.get_id(c, id) == CUDA_SUCCESS;
}

// The array's device address in the current context.  Host code may not use
// g_noalloc_scratch itself: on the host that name is only a stand-in.  The
// first call in a context looks the address up (cudaGetSymbolAddress, which
// also sets the context up if the runtime has not yet); later calls reuse
// it.  Without the driver's context ids every call looks it up.
dvl_status scratch_address(void **out)
{
    unsigned long long id = 0;
    bool have_id = current_ctx_id(&id);
    if (have_id) {
        std::lock_guard<std::mutex> g(g_mu);
        auto it = g_ptr.find(id);
        if (it != g_ptr.end()) {
            *out = it->second;
            return DVL_OK;
        }
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
        return DVL_ERR_CUDA;
    if (!have_id)
        have_id = current_ctx_id(&id);  // the lookup may have made the context
    if (have_id) {
        std::lock_guard<std::mutex> g(g_mu);
        g_ptr[id] = p;
    }
    *out = p;
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
    // The ticket and the best keys must start at zero (every call leaves
    // them so; clearing them again in stream order costs little and repairs
    // a state no call could).  The status word is left alone: its bits
    // accumulate until dvl_noalloc_status reads them.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *base = static_cast<unsigned char *>(scratch);
    if (cudaMemsetAsync(base + dvl::kWsTicket, 0, 4, s) != cudaSuccess ||
        cudaMemsetAsync(base + dvl::kWsBest, 0, kScratchBytes - dvl::kWsBest, s) != cudaSuccess)
        return DVL_ERR_CUDA;
    return dvl_draft_argmax(head, h, M, ids, max_logit, scratch, kScratchBytes, stream);
}

extern "C" dvl_status dvl_noalloc_status(uint32_t *status_bits, void *stream)
{
    if (!status_bits)
        return DVL_ERR_INVALID_ARG;
    void *scratch = nullptr;
    dvl_status st = scratch_address(&scratch);
    if (st != DVL_OK)
        return st;
    // the same read-and-clear as a workspace's status word
    return dvl_workspace_status(scratch, status_bits, stream);
}
