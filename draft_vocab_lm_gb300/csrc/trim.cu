// Load-time trim: gather the rows a ranks list names into a contiguous head.
// ("Masked MTP drafts": drop a ranks .txt next to the model and the head
// weight is trimmed at load; the list's order is kept, so the trimmed head's
// row i is the full head's row ranks[i] and d2t[i] = ranks[i].)
//
// One warp copies one row at a time with 16-byte loads (no L1 allocation)
// and streaming 16-byte stores; rows are handed out grid-stride.  Rows whose
// byte length is not a multiple of 16 fall back to 4-byte copies.
#include <cuda_runtime.h>

#include "dvl_device.cuh"

namespace dvl {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) trim_rows_kernel(const unsigned char *__restrict__ src,
                                                             int64_t row_bytes,
                                                             unsigned char *__restrict__ dst,
                                                             const int32_t *__restrict__ ranks,
                                                             int n)
{
    const int lane = threadIdx.x & 31;
    const long long nw = ((long long)gridDim.x * kThreads) >> 5;
    const long long w0 = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    if ((row_bytes & 15) == 0) {
        const int64_t nv = row_bytes >> 4;
        for (long long i = w0; i < n; i += nw) {
            const uint4 *s = reinterpret_cast<const uint4 *>(src + (int64_t)__ldg(ranks + i) * row_bytes);
            uint4 *d = reinterpret_cast<uint4 *>(dst + (int64_t)i * row_bytes);
#pragma unroll 4
            for (int64_t c = lane; c < nv; c += 32)
                __stcs(d + c, ld_stream16(s + c));
        }
    } else {
        const int64_t nv = row_bytes >> 2;
        for (long long i = w0; i < n; i += nw) {
            const uint32_t *s =
                reinterpret_cast<const uint32_t *>(src + (int64_t)__ldg(ranks + i) * row_bytes);
            uint32_t *d = reinterpret_cast<uint32_t *>(dst + (int64_t)i * row_bytes);
            for (int64_t c = lane; c < nv; c += 32)
                __stcs(d + c, __ldg(s + c));
        }
    }
}

}  // namespace

cudaError_t launch_trim_rows(const unsigned char *src, int64_t src_row_bytes, unsigned char *dst,
                             const int32_t *ranks, int n, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    long long grid = (long long)di.sms * 8;
    const long long need = ((long long)n * 32 + kThreads - 1) / kThreads;
    if (grid > need)
        grid = need;
    if (grid < 1)
        grid = 1;
    trim_rows_kernel<<<(unsigned)grid, kThreads, 0, s>>>(src, src_row_bytes, dst, ranks, n);
    return cudaGetLastError();
}

}  // namespace dvl
