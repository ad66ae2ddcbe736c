// Internal host-side declarations shared by the C ABI and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "dvl.h"

namespace dvl {

// Workspace layout (device bytes).  Every kernel call leaves it as it found
// it: the ticket wraps back to 0 and the best keys are exchanged back to 0.
constexpr int kMaxCtas = 1024;            // grid cap of every reducing kernel
constexpr size_t kWsTicket = 0;           // uint32: blocks finished so far
constexpr size_t kWsStatus = 4;           // uint32: device-side failure bits (1 << dvl_status)
constexpr size_t kWsAmax = 8;             // uint32: a head's max |w| while it is requantized
constexpr size_t kWsBest = 256;           // uint64[DVL_MAX_M]: best key per row (k = 1)
constexpr size_t kWsSlots = 512;          // uint64[M][kMaxCtas][kmax] (k > 1), then
                                          // uint64[M][kMaxGroups][kmax] group lists and
                                          // uint32[kMaxGroups] group tickets
constexpr int kGroup = 16;                // top-k: blocks per first-level merge
constexpr int kMaxGroups = kMaxCtas / kGroup;
constexpr int kTwoLevelLists = 2560;      // top-k merges two-level from M * blocks lists

// Arguments of one reducing launch (one chunk of at most 8 hidden rows).
struct ArgmaxArgs {
    const void *w;            // bf16 [N][K], NVFP4 codes [N][K/2] or FP8 codes [N][K]
    const uint8_t *scales;    // NVFP4 E4M3 [N][K/16]
    float gscale;             // NVFP4 / FP8 tensor scale
    const int32_t *d2t;       // int32 [N] or nullptr
    int64_t id_base;          // full id of row 0 when d2t is null
    int N, K, Kpad;           // Kpad: K rounded up to the kernel's k-step
    const uint16_t *h;        // bf16 [M][K] of this chunk
    int32_t *ids;             // [M][k] of this chunk
    float *logits;            // [M][k] of this chunk
    int k;                    // results per row (1 .. kmax)
    unsigned char *ws;        // workspace base
    bool head_static;         // w / scales / d2t not written by pending work
    int32_t V;                // vocabulary size (<= 2^31 - 1): ids lie in [0, V)
    int32_t m_rows;           // hidden rows of this launch (kernels instantiated for a
                              // padded count read it)
};

// Per-device facts, queried once.
struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};
cudaError_t device_info(DeviceInfo *out);

// Blocks of a streaming kernel that keeps per_sm blocks resident per SM:
// all of them, except that with two or more per SM a few SMs (one in 38, at
// least one) get one block fewer.  Measured on GB300 (152 SMs, so 300
// blocks instead of 304), back-to-back calls: the full 248,320 x 2,560 head
// at one row 178.6 -> 176.2 us, the 32,768 x 5,120 trim at one row 50.7 ->
// 48.9 us and at three rows (register-path MMA) 53.4 -> 51.2 us, the FP8
// full-vocabulary head 94.4 -> 93.3 us.  The gain is about the same number
// of microseconds at every head size: with a few slots free from the start,
// the next call's grid becomes resident (and starts its pre-wait loads)
// while this one runs.
inline long long stream_grid(int sms, int per_sm)
{
    long long g = (long long)sms * per_sm;
    if (per_sm >= 2)
        g -= sms / 38 > 1 ? sms / 38 : 1;
    return g;
}

// Blocks of `func` (launched with `threads` threads and `smem` dynamic shared
// bytes) resident per SM on the current device.  The first query per (kernel,
// device, smem) also raises the kernel's dynamic shared-memory limit; the
// answer is cached.
cudaError_t blocks_per_sm(const void *func, int threads, size_t smem, int *out);

// Launchers (return the launch's cudaError_t).  M is the chunk's row count
// (1 .. 8), kmax is 1 (argmax) or 4 (top-k).
cudaError_t launch_argmax_bf16(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s);
// NVFP4 and FP8 heads (dtype DVL_NVFP4 or DVL_FP8), on the register-path
// tensor cores.
cudaError_t launch_argmax_lowbit(const ArgmaxArgs &a, int dtype, int M, int kmax,
                                 cudaStream_t s);
int max_chunk_rows_bf16(int K);
// Whether a call with M hidden rows (kmax 1: argmax, 4: top-k) runs on the
// register-path tensor cores
// (argmax_bf16_mma.cuh) rather than the CUDA cores (M <= 4) or the tcgen05
// kernel (M >= 5), for a head at w with N rows of width K on a device with
// sms SMs.
bool bf16_uses_mma(const void *w, int N, int K, int M, int kmax, int sms);
// That kernel, for M = 3 .. 16 hidden rows (3 .. 8 at K 5,120 and for top-k).
cudaError_t launch_argmax_bf16_mma(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s);
// Tensor-core argmax / top-k (bf16; kmax 1 or 4) for 5..32 hidden rows in
// one launch.
bool tc_argmax_supported(int M, int K);
cudaError_t launch_argmax_tc(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s);
int max_chunk_rows_lowbit(int K, int kmax);

// The argument checks of draft_argmax / draft_topk, without the workspace.
dvl_status check_reduce_args(const dvl_head *hd, const void *h, int32_t M, int32_t k,
                             const void *ids, const void *logits);

// Arguments of a candidate-scoring launch: out[m][j] = W[ids[m][j] - id_base]
// . h[m] for m < M, j < c (NaN for an id outside the head's N rows).
struct ScoreArgs {
    int dtype;                // DVL_BF16, DVL_NVFP4 or DVL_FP8
    const void *w;            // bf16 [N][K], NVFP4 codes [N][K/2] or FP8 codes [N][K]
    const uint8_t *scales;    // NVFP4 E4M3 [N][K/16]
    float gscale;             // NVFP4 / FP8 tensor scale
    int64_t id_base;          // id of row 0
    int N, K, M, c;
    const uint16_t *h;        // bf16 [M][K]
    const int32_t *ids;       // [M][c]
    float *out;               // [M][c]
};
cudaError_t launch_score(const ScoreArgs &a, cudaStream_t s);

// Requantize a bf16 head of n weights to NVFP4 or FP8 (dtype); reads the
// head's maximum back (synchronizing s) and returns the tensor scale in g_out.
cudaError_t launch_quantize(const uint16_t *w, long long n, int dtype, uint8_t *codes,
                            uint8_t *scales, unsigned char *ws, cudaStream_t s, float *g_out);

cudaError_t launch_trim_rows(const unsigned char *src, int64_t src_row_bytes,
                             unsigned char *dst, const int32_t *ranks, int n,
                             cudaStream_t s);

// Launch `kern` on `s` with programmatic stream serialization allowed, so it
// may begin while the preceding kernel on the stream finishes (the kernel
// itself waits, with griddepcontrol.wait, before it reads that kernel's
// results).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                       const Args &...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace dvl
