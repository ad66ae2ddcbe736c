// Instantiations of the register-path tensor-core kernel for bf16 heads
// (argmax_bf16_mma.cuh) at 9 .. 16 hidden rows, width 2,560, argmax only:
// top-k at those rows runs on tcgen05 (bf16_uses_mma) -- 53.5 against 58.9 us
// at 16 rows on the 52,755-row head.  A translation unit of its own so the
// library builds in parallel.
#include "argmax_bf16_mma.cuh"

namespace dvl {
namespace {

template <int M>
cudaError_t launch_rows(const ArgmaxArgs &a, int kmax, cudaStream_t s)
{
    using namespace bf16mma;
    if (a.K != 2560 || kmax != 1)
        return cudaErrorInvalidValue;
    return launch<M, 1, 2560, 4>(a, s);
}

}  // namespace

cudaError_t launch_argmax_bf16_mma16(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s)
{
    switch (M) {
    case 9: return launch_rows<9>(a, kmax, s);
    case 10: return launch_rows<10>(a, kmax, s);
    case 11: return launch_rows<11>(a, kmax, s);
    case 12: return launch_rows<12>(a, kmax, s);
    case 13: return launch_rows<13>(a, kmax, s);
    case 14: return launch_rows<14>(a, kmax, s);
    case 15: return launch_rows<15>(a, kmax, s);
    case 16: return launch_rows<16>(a, kmax, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dvl
