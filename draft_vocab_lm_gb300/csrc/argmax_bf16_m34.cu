// Instantiations of the bf16 CUDA-core kernel for M in {3, 4} (one
// translation unit per group of M so the library builds in parallel).
#include "argmax_bf16.cuh"

namespace dvl {

cudaError_t launch_argmax_bf16_m34(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s)
{
    using namespace bf16;
    switch (M) {
    case 3: return kmax == 1 ? launch_m<3, 1>(a, s) : launch_m<3, 4>(a, s);
    case 4: return kmax == 1 ? launch_m<4, 1>(a, s) : launch_m<4, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dvl
