// Instantiations and dispatch of the register-path tensor-core kernel for
// bf16 heads (argmax_bf16_mma.cuh): 3 .. 8 hidden rows at widths 2,560 and
// 5,120 here, 9 .. 16 at 2,560 in argmax_bf16_mma16.cu; argmax or top-k.
// The rule that picks it is bf16_uses_mma.
#include "argmax_bf16_mma.cuh"

namespace dvl {
namespace {

template <int M>
cudaError_t launch_rows(const ArgmaxArgs &a, int kmax, cudaStream_t s)
{
    using namespace bf16mma;
    if (a.K == 2560)
        return kmax == 1 ? launch<M, 1, 2560, 4>(a, s) : launch<M, 4, 2560, 4>(a, s);
    if (a.K == 5120)
        return kmax == 1 ? launch<M, 1, 5120, 4>(a, s) : launch<M, 4, 5120, 4>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_argmax_bf16_mma16(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s);

// Up to 16 hidden rows for argmax at K = 2,560.  At 5,120 the staged rows
// leave room for two blocks per SM only up to 8; top-k above 8 rows stays on
// the tcgen05 kernel, whose 138-block grid gives the cross-block merge fewer
// lists (measured at M = 16, 52,755 rows: 55.3 us there against 60.2 us
// here; argmax 45.4 us here against 48.2 us).
bool bf16_uses_mma(const void *w, int N, int K, int M, int kmax, int sms)
{
    const int most = (K == 2560 && kmax == 1) ? bf16mma::kMaxRows : 8;
    return M >= 3 && M <= most && (K == 2560 || K == 5120) &&
           (reinterpret_cast<uintptr_t>(w) & 31) == 0 &&
           (long long)N >= (long long)bf16mma::kTile * bf16mma::kWarps * 2 * sms;
}

cudaError_t launch_argmax_bf16_mma(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s)
{
    switch (M) {
    case 3: return launch_rows<3>(a, kmax, s);
    case 4: return launch_rows<4>(a, kmax, s);
    case 5: return launch_rows<5>(a, kmax, s);
    case 6: return launch_rows<6>(a, kmax, s);
    case 7: return launch_rows<7>(a, kmax, s);
    case 8: return launch_rows<8>(a, kmax, s);
    default: return launch_argmax_bf16_mma16(a, M, kmax, s);
    }
}

}  // namespace dvl
