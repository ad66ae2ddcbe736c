// NVFP4 top-k for 9 .. 32 hidden rows in one pass (16- and 32-row
// instantiations at K = 2,560 and 5,120).
#include "argmax_lowbit.cuh"

namespace dvl {
namespace lowbit {

template cudaError_t launch_groups<kFmtNvfp4, 4>(const ArgmaxArgs &, int, cudaStream_t);

}  // namespace lowbit
}  // namespace dvl
