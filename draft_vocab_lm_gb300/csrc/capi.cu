// The C ABI: argument checks, workspace handling, dispatch to the kernels.
// Every check runs on the host before anything is enqueued.  Nothing here
// allocates or frees device memory, and nothing synchronizes except the two
// calls that read a word back to the host: dvl_quantize_head (the head's
// maximum, at load time) and dvl_workspace_status.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "dvl.h"
#include "dvl_internal.h"

namespace dvl {

namespace {
std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;
std::map<std::tuple<const void *, int, size_t>, int> g_occ;
std::map<std::pair<const void *, int>, size_t> g_smem_limit;  // per kernel and device
thread_local cudaError_t t_last_error = cudaSuccess;

dvl_status cuda_failed(cudaError_t e)
{
    t_last_error = e;
    return DVL_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

cudaError_t device_info(DeviceInfo *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    {
        std::lock_guard<std::mutex> g(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    DeviceInfo di;
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    e = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> g(g_mu);
    g_dev[dev] = di;
    *out = di;
    return cudaSuccess;
}

cudaError_t blocks_per_sm(const void *func, int threads, size_t smem, int *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const auto key = std::make_tuple(func, dev, smem);
    {
        std::lock_guard<std::mutex> g(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    DeviceInfo di;
    e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    if (smem > (size_t)di.smem_optin)
        return cudaErrorInvalidConfiguration;
    {
        // The dynamic shared-memory limit is a property of the kernel, shared
        // by every launch of it: only ever raise it.
        std::lock_guard<std::mutex> g(g_mu);
        size_t &lim = g_smem_limit[std::make_pair(func, dev)];
        if (smem > lim) {
            e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess)
                return e;
            lim = smem;
        }
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> g(g_mu);
    g_occ[key] = n;
    *out = n;
    return cudaSuccess;
}

namespace {

dvl_status check_head(const dvl_head *hd)
{
    if (!hd)
        return DVL_ERR_INVALID_ARG;
    if (hd->dtype != DVL_BF16 && hd->dtype != DVL_NVFP4 && hd->dtype != DVL_FP8)
        return DVL_ERR_INVALID_ARG;
    if ((hd->flags & ~DVL_HEAD_STATIC) != 0 || hd->reserved2 != 0)
        return DVL_ERR_INVALID_ARG;
    if (hd->N < 1 || hd->K < DVL_K_MULTIPLE || hd->K % DVL_K_MULTIPLE != 0 || hd->K > DVL_MAX_K)
        return DVL_ERR_INVALID_ARG;
    if (hd->V < 1 || hd->V > 0x7fffffffLL)
        return DVL_ERR_INVALID_ARG;
    if (!hd->w || !aligned(hd->w, 16))
        return DVL_ERR_INVALID_ARG;
    if (hd->dtype == DVL_NVFP4 && (!hd->scales || !aligned(hd->scales, 16)))
        return DVL_ERR_INVALID_ARG;
    if (hd->dtype != DVL_NVFP4 && hd->scales)
        return DVL_ERR_INVALID_ARG;
    if (hd->d2t) {
        if (!aligned(hd->d2t, 4))
            return DVL_ERR_INVALID_ARG;
    } else if (hd->id_base < 0 || hd->id_base + hd->N > hd->V) {
        return DVL_ERR_INVALID_ARG;
    }
    return DVL_OK;
}

dvl_status reduce_call(const dvl_head *hd, const void *h, int32_t M, int32_t k, int32_t *ids,
                       float *logits, void *ws, size_t ws_bytes, void *stream)
{
    dvl_status st = check_head(hd);
    if (st != DVL_OK)
        return st;
    if (M < 1 || M > DVL_MAX_M || k < 1 || k > DVL_MAX_TOPK || k > hd->N)
        return DVL_ERR_INVALID_ARG;
    if (!h || !aligned(h, 16) || !ids || !aligned(ids, 4) || !logits || !aligned(logits, 4))
        return DVL_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, 16) || ws_bytes < dvl_workspace_bytes(M, k))
        return DVL_ERR_WORKSPACE;
    const int chunk =
        hd->dtype == DVL_BF16 ? max_chunk_rows_bf16(hd->K)
                              : max_chunk_rows_lowbit(hd->K, k == 1 ? 1 : DVL_MAX_TOPK);
    if (chunk < 1)
        return DVL_ERR_UNSUPPORTED;
    ArgmaxArgs a;
    std::memset(&a, 0, sizeof a);
    a.w = hd->w;
    a.scales = hd->scales;
    a.gscale = hd->global_scale;
    a.d2t = hd->d2t;
    a.id_base = hd->id_base;
    a.V = (int32_t)hd->V;
    a.head_static = (hd->flags & DVL_HEAD_STATIC) != 0;
    a.N = hd->N;
    a.K = hd->K;
    a.k = k;
    a.ws = static_cast<unsigned char *>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int kmax = k == 1 ? 1 : DVL_MAX_TOPK;
    if (hd->dtype == DVL_BF16 && M >= 3) {
        DeviceInfo di;
        const cudaError_t e = device_info(&di);
        if (e != cudaSuccess)
            return cuda_failed(e);
        if (bf16_uses_mma(hd->w, hd->N, hd->K, M, kmax, di.sms)) {
            // 3..16 rows on a long head: one pass on the register-path
            // tensor cores
            a.h = static_cast<const uint16_t *>(h);
            a.ids = ids;
            a.logits = logits;
            const cudaError_t el = launch_argmax_bf16_mma(a, M, kmax, s);
            return el == cudaSuccess ? DVL_OK : cuda_failed(el);
        }
    }
    if (hd->dtype == DVL_BF16 && tc_argmax_supported(M, hd->K)) {
        // 5..32 rows: one pass on the tensor cores instead of several
        // CUDA-core passes over the head
        a.h = static_cast<const uint16_t *>(h);
        a.ids = ids;
        a.logits = logits;
        cudaError_t e = launch_argmax_tc(a, M, kmax, s);
        return e == cudaSuccess ? DVL_OK : cuda_failed(e);
    }
    for (int m0 = 0; m0 < M; m0 += chunk) {
        const int mc = M - m0 < chunk ? M - m0 : chunk;
        a.h = static_cast<const uint16_t *>(h) + (size_t)m0 * hd->K;
        a.ids = ids + (size_t)m0 * k;
        a.logits = logits + (size_t)m0 * k;
        cudaError_t e = hd->dtype == DVL_BF16 ? launch_argmax_bf16(a, mc, kmax, s)
                                              : launch_argmax_lowbit(a, hd->dtype, mc, kmax, s);
        if (e != cudaSuccess)
            return cuda_failed(e);
    }
    return DVL_OK;
}

}  // namespace

dvl_status check_reduce_args(const dvl_head *hd, const void *h, int32_t M, int32_t k,
                             const void *ids, const void *logits)
{
    dvl_status st = check_head(hd);
    if (st != DVL_OK)
        return st;
    if (M < 1 || M > DVL_MAX_M || k < 1 || k > DVL_MAX_TOPK || k > hd->N)
        return DVL_ERR_INVALID_ARG;
    if (!h || !aligned(h, 16) || !ids || !aligned(ids, 4) || !logits || !aligned(logits, 4))
        return DVL_ERR_INVALID_ARG;
    return DVL_OK;
}

// The argument checks of a gather into a trimmed head's buffers.
static dvl_status check_gather(const dvl_head *full, void *w_trim, uint8_t *scales_trim,
                               int32_t *d2t)
{
    dvl_status st = check_head(full);
    if (st != DVL_OK)
        return st;
    if ((int64_t)full->N != full->V || full->d2t || full->id_base != 0)
        return DVL_ERR_INVALID_ARG;
    if (!w_trim || !aligned(w_trim, 16) || !d2t || !aligned(d2t, 4))
        return DVL_ERR_INVALID_ARG;
    if (full->dtype == DVL_NVFP4 && (!scales_trim || !aligned(scales_trim, 16)))
        return DVL_ERR_INVALID_ARG;
    return DVL_OK;
}

// Enqueue rows row0 .. row0 + n - 1 of a trimmed head from the full head's
// rows ids[0 .. n - 1] (host ids, already checked), and d2t[row0 + i] =
// ids[i].
static dvl_status enqueue_gather(const dvl_head *full, const int32_t *ids, int32_t n,
                                 int32_t row0, void *w_trim, uint8_t *scales_trim, int32_t *d2t,
                                 void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *d2t_rows = d2t + row0;
    cudaError_t e =
        cudaMemcpyAsync(d2t_rows, ids, (size_t)n * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return cuda_failed(e);
    const int64_t K = full->K;
    const int64_t wrow = full->dtype == DVL_BF16 ? K * 2 : full->dtype == DVL_FP8 ? K : K / 2;
    e = launch_trim_rows(static_cast<const unsigned char *>(full->w), wrow,
                         static_cast<unsigned char *>(w_trim) + (int64_t)row0 * wrow, d2t_rows, n,
                         s);
    if (e == cudaSuccess && full->dtype == DVL_NVFP4)
        e = launch_trim_rows(full->scales, K / 16, scales_trim + (int64_t)row0 * (K / 16),
                             d2t_rows, n, s);
    return e == cudaSuccess ? DVL_OK : cuda_failed(e);
}

// Rows row0 .. row0 + n - 1 of a trimmed head from the full head's rows
// ids[0 .. n - 1] (host ids, checked first), and d2t[row0 + i] = ids[i].
// Repeated ids are counted only when n_duplicates asks for it (a V-byte
// host table, which the load-time trim can afford and a learn need not).
static dvl_status gather_rows(const dvl_head *full, const int32_t *ids, int32_t n,
                              int32_t row0, void *w_trim, uint8_t *scales_trim, int32_t *d2t,
                              int32_t *n_duplicates, void *stream)
{
    dvl_status st = check_gather(full, w_trim, scales_trim, d2t);
    if (st != DVL_OK)
        return st;
    if (!ids || n < 1 || row0 < 0 || (int64_t)row0 + n > 0x7fffffffLL)
        return DVL_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || (int64_t)ids[i] >= full->V)
            return DVL_ERR_OUT_OF_RANGE;
    if (n_duplicates) {
        std::vector<unsigned char> seen((size_t)full->V, 0);
        int32_t dup = 0;
        for (int32_t i = 0; i < n; ++i) {
            dup += seen[(size_t)ids[i]];
            seen[(size_t)ids[i]] = 1;
        }
        *n_duplicates = dup;
    }
    return enqueue_gather(full, ids, n, row0, w_trim, scales_trim, d2t, stream);
}

}  // namespace dvl

using namespace dvl;

extern "C" {

const char *dvl_status_string(int status)
{
    switch (status) {
    case DVL_OK: return "ok";
    case DVL_ERR_INVALID_ARG: return "invalid argument";
    case DVL_ERR_OUT_OF_RANGE: return "id out of range";
    case DVL_ERR_UNSUPPORTED: return "unsupported shape";
    case DVL_ERR_WORKSPACE: return "workspace missing or too small";
    case DVL_ERR_CUDA: return "CUDA error";
    case DVL_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

int dvl_version(void) { return 101; }

size_t dvl_workspace_bytes(int32_t M, int32_t k)
{
    if (M < 1 || M > DVL_MAX_M || k < 1 || k > DVL_MAX_TOPK)
        return 0;
    size_t b = kWsSlots;
    if (k > 1)
        b += (size_t)(kMaxCtas + kMaxGroups) * (size_t)M * DVL_MAX_TOPK * sizeof(uint64_t) +
             (size_t)kMaxGroups * sizeof(uint32_t);
    return b;
}

dvl_status dvl_workspace_init(void *ws, size_t bytes, void *stream)
{
    if (!ws || !aligned(ws, 16) || bytes < kWsSlots)
        return DVL_ERR_WORKSPACE;
    cudaError_t e = cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_failed(e);
    return DVL_OK;
}

dvl_status dvl_workspace_status(void *ws, uint32_t *status_bits, void *stream)
{
    if (!ws || !aligned(ws, 16) || !status_bits)
        return DVL_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *word = static_cast<unsigned char *>(ws) + kWsStatus;
    uint32_t bits = 0u;
    cudaError_t e = cudaMemcpyAsync(&bits, word, sizeof bits, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(word, 0, sizeof bits, s);
    if (e != cudaSuccess)
        return cuda_failed(e);
    *status_bits = bits;
    return DVL_OK;
}

dvl_status dvl_draft_argmax(const dvl_head *head, const void *h, int32_t M, int32_t *ids,
                            float *max_logit, void *ws, size_t ws_bytes, void *stream)
{
    return reduce_call(head, h, M, 1, ids, max_logit, ws, ws_bytes, stream);
}

dvl_status dvl_draft_topk(const dvl_head *head, const void *h, int32_t M, int32_t k,
                          int32_t *ids, float *logits, void *ws, size_t ws_bytes, void *stream)
{
    return reduce_call(head, h, M, k, ids, logits, ws, ws_bytes, stream);
}

dvl_status dvl_draft_plan(const dvl_head *head, int32_t M, int32_t k, const char **kernel,
                          int32_t *launches)
{
    dvl_status st = check_head(head);
    if (st != DVL_OK)
        return st;
    if (M < 1 || M > DVL_MAX_M || k < 1 || k > DVL_MAX_TOPK || k > head->N || !kernel ||
        !launches)
        return DVL_ERR_INVALID_ARG;
    if (head->dtype != DVL_BF16) {
        const int chunk = max_chunk_rows_lowbit(head->K, k == 1 ? 1 : DVL_MAX_TOPK);
        if (chunk < 1)
            return DVL_ERR_UNSUPPORTED;
        *kernel = head->dtype == DVL_NVFP4 ? "nvfp4-mma" : "fp8-mma";
        *launches = (M + chunk - 1) / chunk;
        return DVL_OK;
    }
    if (M >= 3) {
        DeviceInfo di;
        const cudaError_t e = device_info(&di);
        if (e != cudaSuccess)
            return cuda_failed(e);
        if (bf16_uses_mma(head->w, head->N, head->K, M, k == 1 ? 1 : DVL_MAX_TOPK, di.sms)) {
            *kernel = "bf16-mma";
            *launches = 1;
            return DVL_OK;
        }
    }
    if (tc_argmax_supported(M, head->K)) {
        *kernel = "bf16-tcgen05";
        *launches = 1;
        return DVL_OK;
    }
    const int chunk = max_chunk_rows_bf16(head->K);
    if (chunk < 1)
        return DVL_ERR_UNSUPPORTED;
    *kernel = "bf16-cuda-cores";
    *launches = (M + chunk - 1) / chunk;
    return DVL_OK;
}

dvl_status dvl_score_ids(const dvl_head *head, const void *h, int32_t M, const int32_t *ids,
                         int32_t c, float *logits, void *stream)
{
    dvl_status st = check_head(head);
    if (st != DVL_OK)
        return st;
    if (head->d2t || M < 1 || M > DVL_MAX_M || c < 1 || (int64_t)M * c > 0x7fffffffLL)
        return DVL_ERR_INVALID_ARG;
    if (!h || !aligned(h, 16) || !ids || !aligned(ids, 4) || !logits || !aligned(logits, 4))
        return DVL_ERR_INVALID_ARG;
    ScoreArgs a;
    std::memset(&a, 0, sizeof a);
    a.dtype = head->dtype;
    a.w = head->w;
    a.scales = head->scales;
    a.gscale = head->global_scale;
    a.id_base = head->id_base;
    a.N = head->N;
    a.K = head->K;
    a.M = M;
    a.c = c;
    a.h = static_cast<const uint16_t *>(h);
    a.ids = ids;
    a.out = logits;
    cudaError_t e = launch_score(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DVL_OK : cuda_failed(e);
}

dvl_status dvl_trim_head(const dvl_head *full, const int32_t *ranks, int32_t n_ranks,
                         void *w_trim, uint8_t *scales_trim, int32_t *d2t,
                         int32_t *n_duplicates, void *stream)
{
    return gather_rows(full, ranks, n_ranks, 0, w_trim, scales_trim, d2t, n_duplicates, stream);
}

dvl_status dvl_quantize_head(const dvl_head *src, int32_t dtype, void *codes, uint8_t *scales,
                             float *global_scale, void *ws, size_t ws_bytes, void *stream)
{
    dvl_status st = check_head(src);
    if (st != DVL_OK)
        return st;
    if (src->dtype != DVL_BF16 || (dtype != DVL_NVFP4 && dtype != DVL_FP8))
        return DVL_ERR_INVALID_ARG;
    if (!codes || !aligned(codes, 16) || !global_scale)
        return DVL_ERR_INVALID_ARG;
    if ((dtype == DVL_NVFP4) != (scales != nullptr) || (scales && !aligned(scales, 16)))
        return DVL_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, 16) || ws_bytes < dvl_workspace_bytes(1, 1))
        return DVL_ERR_WORKSPACE;
    float g = 1.0f;
    cudaError_t e = launch_quantize(static_cast<const uint16_t *>(src->w),
                                    (long long)src->N * src->K, dtype,
                                    static_cast<uint8_t *>(codes), scales,
                                    static_cast<unsigned char *>(ws),
                                    static_cast<cudaStream_t>(stream), &g);
    if (e != cudaSuccess)
        return cuda_failed(e);
    *global_scale = g;
    return DVL_OK;
}

dvl_status dvl_learn_rows(const dvl_head *full, const int32_t *ids, int32_t n, int32_t row0,
                          void *w_trim, uint8_t *scales_trim, int32_t *d2t, void *stream)
{
    return gather_rows(full, ids, n, row0, w_trim, scales_trim, d2t, nullptr, stream);
}

dvl_status dvl_learn_missing(const dvl_head *full, const int32_t *ids, int32_t n,
                             int32_t *row_of, int32_t *n_rows, int32_t capacity, void *w_trim,
                             uint8_t *scales_trim, int32_t *d2t, int32_t *learned,
                             int32_t *n_learned, void *stream)
{
    dvl_status st = check_gather(full, w_trim, scales_trim, d2t);
    if (st != DVL_OK)
        return st;
    if (n < 0 || (n > 0 && !ids) || !row_of || !n_rows || !learned || !n_learned)
        return DVL_ERR_INVALID_ARG;
    const int32_t row0 = *n_rows;
    if (row0 < 0 || capacity < row0)
        return DVL_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || (int64_t)ids[i] >= full->V)
            return DVL_ERR_OUT_OF_RANGE;  // nothing changed, nothing enqueued
    // first occurrences of ids the list lacks, in order, while rows remain
    int32_t m = 0;
    for (int32_t i = 0; i < n && row0 + m < capacity; ++i) {
        const int32_t t = ids[i];
        if (row_of[t] >= 0)
            continue;
        row_of[t] = row0 + m;  // also skips later repeats of t
        learned[m++] = t;
    }
    *n_learned = m;
    if (m == 0)
        return DVL_OK;
    st = enqueue_gather(full, learned, m, row0, w_trim, scales_trim, d2t, stream);
    if (st != DVL_OK) {
        for (int32_t i = 0; i < m; ++i)
            row_of[learned[i]] = -1;  // undo: the rows were not written
        *n_learned = 0;
        return st;
    }
    *n_rows = row0 + m;
    return DVL_OK;
}

const char *dvl_last_error(void) { return cudaGetErrorString(t_last_error); }

}  // extern "C"
