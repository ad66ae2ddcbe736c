// FP8 argmax / top-k with the hidden width read at run time.
#include "argmax_lowbit.cuh"

namespace dvl {
namespace lowbit {

template cudaError_t launch_rt<kFmtFp8>(const ArgmaxArgs &, int, int, cudaStream_t);

}  // namespace lowbit
}  // namespace dvl
