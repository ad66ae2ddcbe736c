// Dispatch of the NVFP4 argmax / top-k kernel (argmax_nvfp4.cuh) to its
// instantiations.
#include "argmax_nvfp4.cuh"

namespace dvl {

cudaError_t launch_argmax_nvfp4_kc(const ArgmaxArgs &a, int M, cudaStream_t s);
cudaError_t launch_argmax_nvfp4_rt(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s);

// Hidden rows per launch: up to 8 (one MMA n8 tile), and few enough that the
// staged hidden rows leave room for two blocks per SM; 0 if not even one fits.
int max_chunk_rows_nvfp4(int K)
{
    const int Kpad = nvfp4::kpad_of(K);
    for (int M = 8; M >= 1; --M)
        if (nvfp4::nvfp4_h_bytes(Kpad, M) + (size_t)M * nvfp4::kLists * 4 * 8 <= 110 * 1024)
            return M;
    return 0;
}

cudaError_t launch_argmax_nvfp4(const ArgmaxArgs &a_in, int M, int kmax, cudaStream_t s)
{
    ArgmaxArgs a = a_in;
    a.Kpad = nvfp4::kpad_of(a.K);
    // argmax at the unrolled widths: one base pointer per group with
    // immediate offsets (measured 29.0 -> 20.4 us on a 32k x 5,120 head)
    if (kmax == 1 && M <= 4 && (a.K == 5120 || a.K == 2560))
        return launch_argmax_nvfp4_kc(a, M, s);
    return launch_argmax_nvfp4_rt(a, M, kmax, s);
}

}  // namespace dvl
