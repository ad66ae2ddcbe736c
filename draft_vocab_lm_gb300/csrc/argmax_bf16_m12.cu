// Instantiations of the bf16 CUDA-core kernel for M in {1, 2} (one
// translation unit per group of M so the library builds in parallel).
#include "argmax_bf16.cuh"

namespace dvl {

cudaError_t launch_argmax_bf16_m12(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s)
{
    using namespace bf16;
    switch (M) {
    case 1: return kmax == 1 ? launch_m<1, 1>(a, s) : launch_m<1, 4>(a, s);
    case 2: return kmax == 1 ? launch_m<2, 1>(a, s) : launch_m<2, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dvl
