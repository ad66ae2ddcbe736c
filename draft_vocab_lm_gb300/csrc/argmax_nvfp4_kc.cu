// NVFP4 argmax with the hidden width unrolled at compile time (K = 2,560 and
// 5,120, up to 4 hidden rows per launch).
#include "argmax_nvfp4.cuh"

namespace dvl {

cudaError_t launch_argmax_nvfp4_kc(const ArgmaxArgs &a, int M, cudaStream_t s)
{
    using namespace nvfp4;
    if (a.K == 5120) {
        switch (M) {
        case 1: return launch_one<1, 1, 5120>(a, s);
        case 2: return launch_one<2, 1, 5120>(a, s);
        case 3: return launch_one<3, 1, 5120>(a, s);
        case 4: return launch_one<4, 1, 5120>(a, s);
        }
    } else if (a.K == 2560) {
        switch (M) {
        case 1: return launch_one<1, 1, 2560>(a, s);
        case 2: return launch_one<2, 1, 2560>(a, s);
        case 3: return launch_one<3, 1, 2560>(a, s);
        case 4: return launch_one<4, 1, 2560>(a, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace dvl
