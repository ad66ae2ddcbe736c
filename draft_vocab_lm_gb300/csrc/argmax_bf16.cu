// Dispatch of the bf16 CUDA-core argmax / top-k kernel (argmax_bf16.cuh) to
// its per-M instantiations.
#include "argmax_bf16.cuh"

namespace dvl {

cudaError_t launch_argmax_bf16_m12(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s);
cudaError_t launch_argmax_bf16_m34(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s);

// Hidden rows per launch: at most 4 (argmax at 5 or more rows runs on the
// tensor cores; top-k at 5 or more rows runs in chunks of 4), and the fp32
// copy of the chunk in shared memory stays within 96 KB so two blocks fit on
// an SM.
int max_chunk_rows_bf16(int K)
{
    int r = (96 * 1024) / (bf16::kpad_of(K) * 4);
    return r > 4 ? 4 : r;
}

cudaError_t launch_argmax_bf16(const ArgmaxArgs &a_in, int M, int kmax, cudaStream_t s)
{
    ArgmaxArgs a = a_in;
    a.Kpad = bf16::kpad_of(a.K);
    if (M <= 2)
        return launch_argmax_bf16_m12(a, M, kmax, s);
    return launch_argmax_bf16_m34(a, M, kmax, s);
}

}  // namespace dvl
