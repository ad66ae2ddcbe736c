// Dispatch of the low-bit (NVFP4, FP8) argmax / top-k kernel
// (argmax_lowbit.cuh) to its instantiations.
#include "argmax_lowbit.cuh"

namespace dvl {

// Hidden rows per launch.  At the unrolled widths: 32 at 2,560 for argmax,
// 16 otherwise (up to four groups of 8 MMA columns; 32 rows of top-k lists
// next to 32 staged rows would not fit in shared memory).  Other widths: up
// to 8 (one MMA n8 tile), and few enough that the staged hidden rows leave
// room for two blocks per SM; 0 if not even one fits.
int max_chunk_rows_lowbit(int K, int kmax)
{
    if (K == 2560)
        return kmax == 1 ? 32 : 16;
    if (K == 5120)
        return 16;
    const int Kpad = lowbit::kpad_of(K);
    for (int M = 8; M >= 1; --M)
        if (lowbit::lowbit_h_bytes(Kpad, M) + (size_t)M * lowbit::kLists * 4 * 8 <= 110 * 1024)
            return M;
    return 0;
}

cudaError_t launch_argmax_lowbit(const ArgmaxArgs &a_in, int dtype, int M, int kmax,
                                 cudaStream_t s)
{
    using namespace lowbit;
    ArgmaxArgs a = a_in;
    a.Kpad = kpad_of(a.K);
    // argmax and top-k at the unrolled widths: one base pointer per group
    // with immediate offsets (measured 29.0 -> 20.4 us on a 32k x 5,120 NVFP4
    // head)
    const bool kc = M <= 4 && (a.K == 5120 || a.K == 2560);
    // 9 .. 32 rows at the unrolled widths: one pass over the head
    const bool groups = M > 8 && (a.K == 5120 || a.K == 2560);
    if (dtype == DVL_NVFP4) {
        if (kc)
            return kmax == 1 ? launch_kc<kFmtNvfp4, 1>(a, M, s) : launch_kc<kFmtNvfp4, 4>(a, M, s);
        if (groups)
            return kmax == 1 ? launch_groups<kFmtNvfp4, 1>(a, M, s)
                             : launch_groups<kFmtNvfp4, 4>(a, M, s);
        return launch_rt<kFmtNvfp4>(a, M, kmax, s);
    }
    if (dtype == DVL_FP8) {
        if (kc)
            return kmax == 1 ? launch_kc<kFmtFp8, 1>(a, M, s) : launch_kc<kFmtFp8, 4>(a, M, s);
        if (groups)
            return kmax == 1 ? launch_groups<kFmtFp8, 1>(a, M, s) : launch_groups<kFmtFp8, 4>(a, M, s);
        return launch_rt<kFmtFp8>(a, M, kmax, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dvl
