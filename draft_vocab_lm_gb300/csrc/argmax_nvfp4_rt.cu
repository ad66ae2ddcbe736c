// NVFP4 argmax / top-k with the hidden width read at run time.
#include "argmax_nvfp4.cuh"

namespace dvl {

cudaError_t launch_argmax_nvfp4_rt(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s)
{
    using namespace nvfp4;
    return kmax == 1 ? dispatch_m<1, 0>(a, M, s) : dispatch_m<4, 0>(a, M, s);
}

}  // namespace dvl
