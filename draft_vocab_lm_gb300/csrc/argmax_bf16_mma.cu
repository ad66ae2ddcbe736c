// Instantiations and dispatch of the register-path tensor-core kernel for
// bf16 heads (argmax_bf16_mma.cuh): 3 .. 8 hidden rows, widths 2,560 and
// 5,120, argmax or top-k.  The rule that picks it is bf16_uses_mma.
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

bool bf16_uses_mma(const void *w, int N, int K, int M, int sms)
{
    return M >= 3 && M <= bf16mma::kMaxRows && (K == 2560 || K == 5120) &&
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
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dvl
